// Attention of a few query rows per head over the KV rows a page / block table selects, read in place.
//
// CompactAttention, 'Method steps' (3): the per-group KV block list T[b,g] (kv_indptr / kv_indices)
// is handed to a paged dense-attention kernel that reads the selected blocks of the KV-head-major
// cache where they are, with no copy; DELTA, 'Overall framework': sparse layers attend only over the
// selected page set.  Each (sequence, layer, KV head) row of the table serves the G query heads of
// its group, n_q query rows each (R = G * n_q rows), with no causal mask (decode-style queries come
// after every selected key).
//
// Split-K: the blocks of a row are divided among S CTAs; each CTA walks its blocks in chunks of up to
// 128 cache rows staged in shared memory, keeps an online (max, sum) and the weighted V sum per query
// row, and writes a partial; attend_combine merges the S partials of each query row.
#include "internal.cuh"

namespace kvsel {
namespace {

constexpr int kAttThreads = 256;
constexpr int kChunk = 128;          // cache rows per shared-memory chunk
constexpr int kMaxR = 32;            // query rows per table row
constexpr int kRowPad = 8;           // bf16 elements of padding per staged row

struct AttArgs {
  const __nv_bfloat16* q;
  const uint4* k;
  const uint4* v;
  const int32_t* indptr;      // nullable
  const int32_t* indices;     // nullable (then every block of the row's cache, in order)
  float* part;                // [rows][S][R][d + 2]: acc[d], m, l
  float* o;                   // [batch][n_layers][h_q][n_q][d]
  DeviceError* err;           // a block id outside the cache is skipped and recorded here
  int32_t n_layers, h_q, h_kv, d, G, n_q, R, P, n_per_row, S;
  float scale_log2;
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Block list of table row r: [beg, end) into `indices` (or the implicit list 0 .. n_blocks - 1).
__device__ __forceinline__ void row_list(const AttArgs& a, const SeqInfo& si, int r, int& beg, int& end) {
  if (a.indices == nullptr) {
    beg = 0;
    end = (si.n_keys + a.P - 1) / a.P;
  } else if (a.indptr == nullptr) {
    beg = r * a.n_per_row;
    end = beg + a.n_per_row;
  } else {
    beg = a.indptr[r];
    end = a.indptr[r + 1];
  }
}

template <int D>
__global__ void __launch_bounds__(kAttThreads) attend_split(const __grid_constant__ AttArgs a,
                                                            const __grid_constant__ SeqTable t) {
  constexpr int LDR = D + kRowPad;                 // staged row stride (bf16)
  constexpr int VPR = D / 8;                       // 16-byte vectors per row
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  __nv_bfloat16* Vs = Ks + kChunk * LDR;
  float* Qs = reinterpret_cast<float*>(Vs + kChunk * LDR);        // [R][D], pre-scaled by log2(e)/sqrt(d)
  float* Ps = Qs + kMaxR * D;                                      // [R][kChunk] logits, then weights
  float* Mr = Ps + kMaxR * kChunk;                                 // running max per row
  float* Lr = Mr + kMaxR;                                          // running sum per row
  float* Fr = Lr + kMaxR;                                          // rescale factor of this chunk
  int32_t* src = reinterpret_cast<int32_t*>(Fr + kMaxR);           // cache row of each staged row

  const int tid = threadIdx.x;
  const int r = blockIdx.x / a.S, s = blockIdx.x % a.S;
  const int per_seq = a.n_layers * a.h_kv;
  const int b = r / per_seq, lg = r % per_seq;
  const int layer = lg / a.h_kv, g = lg % a.h_kv;
  const SeqInfo& si = t.s[b];
  int beg, end;
  row_list(a, si, r, beg, end);
  const int nb = end - beg;
  const int b0 = beg + (int)(((int64_t)s * nb) / a.S), b1 = beg + (int)(((int64_t)(s + 1) * nb) / a.S);
  const uint4* kbase = a.k + si.k_off / 8 + ((int64_t)layer * a.h_kv + g) * si.n_keys * VPR;
  const uint4* vbase = a.v + si.k_off / 8 + ((int64_t)layer * a.h_kv + g) * si.n_keys * VPR;

  // query rows j = h_local * n_q + i of the group, in fp32, scaled for base-2 exponentials
  for (int x = tid; x < a.R * D; x += kAttThreads) {
    const int j = x / D, c = x % D;
    const int h = g * a.G + j / a.n_q, i = j % a.n_q;
    const int64_t off = ((((int64_t)b * a.n_layers + layer) * a.h_q + h) * a.n_q + i) * D + c;
    Qs[x] = __bfloat162float(a.q[off]) * a.scale_log2;
  }
  if (tid < kMaxR) {
    Mr[tid] = -INFINITY;
    Lr[tid] = 0.f;
  }
  // PV ownership: (row j, dim pair) items, R * D / 2 of them over the threads
  constexpr int kPairs = D / 2;
  const int n_items = a.R * kPairs;
  float2 acc[(kMaxR * kPairs + kAttThreads - 1) / kAttThreads];
#pragma unroll
  for (int u = 0; u < (int)(sizeof(acc) / sizeof(acc[0])); ++u) acc[u] = make_float2(0.f, 0.f);

  int blk = b0;          // next block to stage
  int within = 0;        // next row inside it
  while (blk < b1) {
    __syncthreads();     // the previous chunk is consumed
    // table of this chunk's cache rows (one thread walks the blocks: chunks are short)
    if (tid == 0) {
      int n = 0;
      while (n < kChunk && blk < b1) {
        const int id = a.indices == nullptr ? blk : a.indices[blk];
        const int64_t row = (int64_t)id * a.P + within;
        if (id >= 0 && row < si.n_keys) src[n++] = (int32_t)row;
        else if (within == 0) set_device_error(a.err, KVSEL_ERR_DEVICE, (uint32_t)blk);   // no row of the block exists
        if (++within == a.P || row + 1 >= si.n_keys || id < 0) {
          within = 0;
          ++blk;
        }
      }
      src[kChunk] = n;
      src[kChunk + 1] = blk;
      src[kChunk + 2] = within;
    }
    __syncthreads();
    const int n = src[kChunk];
    blk = src[kChunk + 1];
    within = src[kChunk + 2];
    // stage K and V rows (16-byte vectors; consecutive threads take consecutive vectors of a row)
    for (int x = tid; x < n * VPR; x += kAttThreads) {
      const int rr = x / VPR, c = x % VPR;
      const int64_t row = src[rr];
      *reinterpret_cast<uint4*>(Ks + rr * LDR + c * 8) = kbase[row * VPR + c];
      *reinterpret_cast<uint4*>(Vs + rr * LDR + c * 8) = vbase[row * VPR + c];
    }
    __syncthreads();
    // logits: thread pair (key, half) computes R dot products over D / 2 dims; the loop bound is
    // uniform over each warp (the pair sum is a shuffle), rows past n compute on row 0 and are dropped
    for (int xb = 0; xb < 2 * n; xb += kAttThreads) {
      const int x = xb + tid;
      const bool valid = x < 2 * n;
      const int key = valid ? (x >> 1) : 0, half = x & 1;
      float kf[D / 2];
#pragma unroll
      for (int c = 0; c < D / 16; ++c)
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(Ks + key * LDR + half * (D / 2) + c * 8), kf + c * 8);
      for (int j = 0; j < a.R; ++j) {
        const float* qj = Qs + j * D + half * (D / 2);
        float z = 0.f;
#pragma unroll
        for (int c = 0; c < D / 2; ++c) z = fmaf(qj[c], kf[c], z);
        z += __shfl_xor_sync(0xffffffffu, z, 1);
        if (valid && half == 0) Ps[j * kChunk + key] = z;
      }
    }
    __syncthreads();
    // online softmax per query row: one warp per row
    for (int j = tid >> 5; j < a.R; j += kAttThreads / 32) {
      const int lane = tid & 31;
      float mx = -INFINITY;
      for (int x = lane; x < n; x += 32) mx = fmaxf(mx, Ps[j * kChunk + x]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_old = Mr[j];
      const float m_new = fmaxf(m_old, mx);
      float sum = 0.f;
      for (int x = lane; x < n; x += 32) {
        const float p = fast_ex2(Ps[j * kChunk + x] - m_new);
        Ps[j * kChunk + x] = p;
        sum += p;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) {
        const float f = m_old == -INFINITY ? 0.f : fast_ex2(m_old - m_new);
        Fr[j] = f;
        Lr[j] = Lr[j] * f + sum;
        Mr[j] = m_new;
      }
    }
    __syncthreads();
    // weighted V sum: each thread owns (row, dim pair) items
#pragma unroll
    for (int u = 0; u < (int)(sizeof(acc) / sizeof(acc[0])); ++u) {
      const int item = tid + u * kAttThreads;
      if (item < n_items) {
        const int j = item / kPairs, pr = item % kPairs;
        const float f = Fr[j];
        float2 s2 = make_float2(acc[u].x * f, acc[u].y * f);
        const float* pj = Ps + j * kChunk;
        for (int x = 0; x < n; ++x) {
          const __nv_bfloat162 vv = *reinterpret_cast<const __nv_bfloat162*>(Vs + x * LDR + 2 * pr);
          const float2 vf = __bfloat1622float2(vv);
          s2.x = fmaf(pj[x], vf.x, s2.x);
          s2.y = fmaf(pj[x], vf.y, s2.y);
        }
        acc[u] = s2;
      }
    }
  }
  __syncthreads();
  // partial of this split: acc[d], m, l per query row
  float* out = a.part + ((int64_t)r * a.S + s) * a.R * (D + 2);
#pragma unroll
  for (int u = 0; u < (int)(sizeof(acc) / sizeof(acc[0])); ++u) {
    const int item = tid + u * kAttThreads;
    if (item < n_items) {
      const int j = item / kPairs, pr = item % kPairs;
      out[j * (D + 2) + 2 * pr] = acc[u].x;
      out[j * (D + 2) + 2 * pr + 1] = acc[u].y;
    }
  }
  if (tid < a.R) {
    out[tid * (D + 2) + D] = Mr[tid];
    out[tid * (D + 2) + D + 1] = Lr[tid];
  }
}

// Decode-sized groups (R <= 8 query rows per table row): one warp per split, no block-wide
// synchronisation in the loop.  A step covers 16 key positions of the split: the lanes copy the
// step's K and V rows into the warp's shared-memory stage with cp.async (whole rows per copy
// instruction; zero-filled where a position selects no row), and the next step's copies are issued
// before this step's arithmetic.  Lane i takes key i % 16 and half i / 16 of the head dim for the
// logits (K chunks XOR-swizzled by the key, so the lanes' reads hit distinct banks; query rows read
// from shared memory as broadcasts), the online softmax runs across the 16 keys with shuffles, and in
// the weighted V sum lane i owns dims DPL*i .. DPL*i + DPL - 1.  Small stages keep 12 warps per SM.
constexpr int kWarpsPerCta = 4;
constexpr int kStep = 16;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const uint32_t n = valid ? 16u : 0u;   // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int D, int R>
__global__ void __launch_bounds__(32 * kWarpsPerCta) attend_warp(const __grid_constant__ AttArgs a,
                                                                 const __grid_constant__ SeqTable t) {
  constexpr int VPR = D / 8;          // 16-byte chunks per row
  constexpr int DPL = D / 32;         // dims per lane in the V sum
  constexpr int STAGE = kStep * D;    // bf16 elements of one K (or V) stage
  constexpr int HC = VPR / 2;         // chunks per half row
  extern __shared__ __align__(16) uint8_t smem_raw[];
  float* Qs = reinterpret_cast<float*>(smem_raw);                                   // [R][D]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __nv_bfloat16* Kb = reinterpret_cast<__nv_bfloat16*>(smem_raw + R * D * 4) + warp * 4 * STAGE;   // [2][16][D]
  __nv_bfloat16* Vb = Kb + 2 * STAGE;                                                              // [2][16][D]
  const int per_cta = a.S / kWarpsPerCta;
  const int r = blockIdx.x / per_cta;
  const int s = (blockIdx.x % per_cta) * kWarpsPerCta + warp;
  const int per_seq = a.n_layers * a.h_kv;
  const int b = r / per_seq, lg = r % per_seq;
  const int layer = lg / a.h_kv, g = lg % a.h_kv;
  const SeqInfo& si = t.s[b];
  // query rows j < a.R of the group (rows up to the template's R beyond them are zero and unused)
  for (int x = threadIdx.x; x < R * D; x += 32 * kWarpsPerCta) {
    const int j = x / D, c = x % D;
    float qv = 0.f;
    if (j < a.R) {
      const int h = g * a.G + j / a.n_q, i = j % a.n_q;
      const int64_t off = ((((int64_t)b * a.n_layers + layer) * a.h_q + h) * a.n_q + i) * D + c;
      qv = __bfloat162float(a.q[off]) * a.scale_log2;
    }
    Qs[x] = qv;
  }
  __syncthreads();
  int beg, end;
  row_list(a, si, r, beg, end);
  const int64_t n_pos = (int64_t)(end - beg) * a.P;                  // key positions of the row
  const int64_t p0 = (s * n_pos) / a.S, p1 = ((s + 1) * n_pos) / a.S;
  const __nv_bfloat16* kbase =
      reinterpret_cast<const __nv_bfloat16*>(a.k) + si.k_off + ((int64_t)layer * a.h_kv + g) * si.n_keys * D;
  const __nv_bfloat16* vbase =
      reinterpret_cast<const __nv_bfloat16*>(a.v) + si.k_off + ((int64_t)layer * a.h_kv + g) * si.n_keys * D;
  const uint32_t kb_s = (uint32_t)__cvta_generic_to_shared(Kb), vb_s = (uint32_t)__cvta_generic_to_shared(Vb);
  const int key = lane & (kStep - 1), half = lane >> 4;

  // Block id of this lane's key position (fetched a step ahead of its use), and its cache row or -1.
  auto id_at = [&](int64_t pos) -> int32_t {
    if (pos >= p1) return -1;
    const int bi = (int)(pos / a.P);
    return a.indices == nullptr ? bi : __ldg(a.indices + beg + bi);
  };
  auto row_of = [&](int64_t pos, int32_t id) -> int32_t {
    if (pos >= p1) return -1;
    const int bi = (int)(pos / a.P), within = (int)(pos - (int64_t)bi * a.P);
    const int64_t rr = (int64_t)id * a.P + within;
    if (id >= 0 && rr < si.n_keys) return (int32_t)rr;
    if (within == 0 && half == 0) set_device_error(a.err, KVSEL_ERR_DEVICE, (uint32_t)(beg + bi));
    return -1;
  };
  // Copy of one stage: lane takes 16-byte chunk lane % VPR of key lane / VPR + (32 / VPR) * i, so each
  // copy instruction reads whole rows (512 contiguous bytes per two rows at d = 128).
  auto issue = [&](int32_t row, int buf) {
    constexpr int KPI = 32 / VPR;                   // keys per instruction
    const int c = lane % VPR;
#pragma unroll
    for (int i = 0; i < kStep / KPI; ++i) {
      const int x = i * KPI + lane / VPR;
      const int32_t rx = __shfl_sync(0xffffffffu, row, x);
      const int64_t src = (int64_t)(rx < 0 ? 0 : rx) * D + c * 8;
      const uint32_t kd = kb_s + (uint32_t)((buf * STAGE + x * D) * 2 + ((c ^ (x & (VPR - 1))) * 16));
      const uint32_t vd = vb_s + (uint32_t)((buf * STAGE + x * D) * 2 + c * 16);
      cp_async16(kd, kbase + src, rx >= 0);
      cp_async16(vd, vbase + src, rx >= 0);
    }
    cp_async_commit();
  };

  float m[R], l[R], acc[R][DPL];
#pragma unroll
  for (int j = 0; j < R; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int c = 0; c < DPL; ++c) acc[j][c] = 0.f;
  }
  int32_t row = row_of(p0 + key, id_at(p0 + key));
  int32_t id_next = id_at(p0 + kStep + key);
  if (p0 < p1) issue(row, 0);
  int buf = 0;
  for (int64_t base = p0; base < p1; base += kStep) {
    const bool more = base + kStep < p1;
    int32_t row_next = -1;
    const int32_t id_after = id_at(base + 2 * kStep + key);
    if (more) {
      row_next = row_of(base + kStep + key, id_next);
      issue(row_next, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    id_next = id_after;
    __syncwarp();
    // logits: this lane's key, half of the head dim, two partial sums per row for ILP
    const __nv_bfloat16* krow = Kb + buf * STAGE + key * D;
    float z[R], z2[R];
#pragma unroll
    for (int j = 0; j < R; ++j) z[j] = z2[j] = 0.f;
#pragma unroll
    for (int cc = 0; cc < HC; ++cc) {
      const int c = half * HC + cc;
      float kf[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(krow + ((c ^ (key & (VPR - 1))) * 8)), kf);
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const float4 q0 = *reinterpret_cast<const float4*>(Qs + j * D + c * 8);
        const float4 q1 = *reinterpret_cast<const float4*>(Qs + j * D + c * 8 + 4);
        z[j] = fmaf(q0.x, kf[0], fmaf(q0.y, kf[1], fmaf(q0.z, kf[2], fmaf(q0.w, kf[3], z[j]))));
        z2[j] = fmaf(q1.x, kf[4], fmaf(q1.y, kf[5], fmaf(q1.z, kf[6], fmaf(q1.w, kf[7], z2[j]))));
      }
    }
    // online softmax across the 16 keys of the step (both halves hold the same values)
    float p[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
      float zj = z[j] + z2[j];
      zj += __shfl_xor_sync(0xffffffffu, zj, 16);
      zj = row >= 0 ? zj : -INFINITY;
      float mx = zj;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m[j], mx);
      const float f = m[j] == -INFINITY ? 0.f : fast_ex2(m[j] - m_new);
      p[j] = m_new == -INFINITY ? 0.f : fast_ex2(zj - m_new);
      float sum = p[j];
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      l[j] = l[j] * f + sum;
      m[j] = m_new;
#pragma unroll
      for (int c = 0; c < DPL; ++c) acc[j][c] *= f;
    }
    // weighted V sum over the 16 keys (zero-filled rows carry p = 0)
    const __nv_bfloat16* vst = Vb + buf * STAGE + DPL * lane;
#pragma unroll
    for (int x = 0; x < kStep; ++x) {
      float vf[DPL];
      if constexpr (DPL == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(vst + x * D);
        vf[0] = __uint_as_float(u.x << 16);
        vf[1] = __uint_as_float(u.x & 0xffff0000u);
        vf[2] = __uint_as_float(u.y << 16);
        vf[3] = __uint_as_float(u.y & 0xffff0000u);
      } else {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(vst + x * D);
        vf[0] = __uint_as_float(u << 16);
        vf[1] = __uint_as_float(u & 0xffff0000u);
      }
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const float px = __shfl_sync(0xffffffffu, p[j], x);
#pragma unroll
        for (int c = 0; c < DPL; ++c) acc[j][c] = fmaf(px, vf[c], acc[j][c]);
      }
    }
    __syncwarp();          // the stage is read before it is refilled
    row = row_next;
    buf ^= 1;
  }
  float* out = a.part + ((int64_t)r * a.S + s) * a.R * (D + 2);
#pragma unroll
  for (int j = 0; j < R; ++j) {
    if (j >= a.R) break;
#pragma unroll
    for (int c = 0; c < DPL; ++c) out[j * (D + 2) + DPL * lane + c] = acc[j][c];
    if (lane == 0) {
      out[j * (D + 2) + D] = m[j];
      out[j * (D + 2) + D + 1] = l[j];
    }
  }
}

size_t attend_warp_smem(int d, int R) {
  return (size_t)R * d * 4 + (size_t)kWarpsPerCta * 4 * kStep * d * 2;
}

// o[row j of table row r] = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s; rows with no key give 0.
template <int D>
__global__ void __launch_bounds__(D) attend_combine(const __grid_constant__ AttArgs a) {
  __shared__ float ms[256], ws_[256];
  const int rj = blockIdx.x;
  const int r = rj / a.R, j = rj % a.R;
  const int c = threadIdx.x;
  const float* p = a.part + (int64_t)r * a.S * a.R * (D + 2) + j * (D + 2);
  const int64_t stride = (int64_t)a.R * (D + 2);
  // the splits' maxima and sums, loaded in parallel
  for (int s = c; s < a.S; s += D) {
    ms[s] = p[s * stride + D];
    ws_[s] = p[s * stride + D + 1];
  }
  __syncthreads();
  float M = -INFINITY;
  for (int s = 0; s < a.S; ++s) M = fmaxf(M, ms[s]);
  float num = 0.f, den = 0.f;
  if (M > -INFINITY) {
#pragma unroll 4
    for (int s = 0; s < a.S; ++s) {
      const float m = ms[s];
      const float w = m == -INFINITY ? 0.f : exp2f(m - M);
      num = fmaf(w, p[s * stride + c], num);
      den = fmaf(w, ws_[s], den);
    }
  }
  const int per_seq = a.n_layers * a.h_kv;
  const int b = r / per_seq, lg = r % per_seq;
  const int layer = lg / a.h_kv, g = lg % a.h_kv;
  const int h = g * a.G + j / a.n_q, i = j % a.n_q;
  const int64_t off = ((((int64_t)b * a.n_layers + layer) * a.h_q + h) * a.n_q + i) * D + c;
  a.o[off] = den > 0.f ? num / den : 0.f;
}

}  // namespace

int64_t attend_splits(int64_t rows, int64_t max_rows_per_list, int R) {
  if (R <= 8) {
    // warp splits: about 4096 warps over the GPU, no split shorter than 64 positions; a multiple of
    // the warps per CTA
    int64_t s = (4096 + rows - 1) / rows;
    const int64_t cap = (max_rows_per_list + 63) / 64;
    if (s > cap) s = cap;
    s = (s + kWarpsPerCta - 1) / kWarpsPerCta * kWarpsPerCta;
    if (s < kWarpsPerCta) s = kWarpsPerCta;
    if (s > 256) s = 256;
    return s;
  }
  // block splits: enough CTAs to fill the GPU a few times over, no split shorter than one chunk
  int64_t s = (2048 + rows - 1) / rows;
  const int64_t cap = (max_rows_per_list + kChunk - 1) / kChunk;
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  return s;
}

size_t attend_smem(int d) {
  return sizeof(__nv_bfloat16) * 2 * (size_t)kChunk * (d + kRowPad) +
         sizeof(float) * ((size_t)kMaxR * d + (size_t)kMaxR * kChunk + 3 * kMaxR) + sizeof(int32_t) * (kChunk + 3);
}

kvsel_status launch_attend(const kvsel_desc& d, const SeqTable& t, const void* q, int n_q, const void* k,
                           const void* v, const int32_t* indptr, const int32_t* indices, int n_per_row, int P,
                           int64_t S, float* part, float* o, DeviceError* err, cudaStream_t s) {
  AttArgs a;
  a.err = err;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const uint4*>(k);
  a.v = static_cast<const uint4*>(v);
  a.indptr = indptr;
  a.indices = indices;
  a.part = part;
  a.o = o;
  a.n_layers = d.n_layers;
  a.h_q = d.h_q;
  a.h_kv = d.h_kv;
  a.d = d.head_dim;
  a.G = d.h_q / d.h_kv;
  a.n_q = n_q;
  a.R = a.G * n_q;
  a.P = P;
  a.n_per_row = n_per_row;
  a.S = (int32_t)S;
  a.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)d.head_dim));
  const int64_t rows = (int64_t)d.batch * d.n_layers * d.h_kv;
  const size_t smem = attend_smem(d.head_dim);
  kvsel_status st;
  if (a.R <= 8) {
    TraceScope ts("attend_split", s);
    const unsigned grid = (unsigned)(rows * S / kWarpsPerCta);
    const int Rt = a.R == 1 ? 1 : a.R == 2 ? 2 : a.R <= 4 ? 4 : 8;
    const size_t wsm = attend_warp_smem(d.head_dim, Rt);
    cudaError_t ce = cudaSuccess;
    auto go = [&](auto kern) {
      if ((ce = set_smem((const void*)kern, wsm)) == cudaSuccess) kern<<<grid, 32 * kWarpsPerCta, wsm, s>>>(a, t);
    };
    if (d.head_dim == 64) {
      if (a.R == 1) go(attend_warp<64, 1>);
      else if (a.R == 2) go(attend_warp<64, 2>);
      else if (a.R <= 4) go(attend_warp<64, 4>);
      else go(attend_warp<64, 8>);
    } else {
      if (a.R == 1) go(attend_warp<128, 1>);
      else if (a.R == 2) go(attend_warp<128, 2>);
      else if (a.R <= 4) go(attend_warp<128, 4>);
      else go(attend_warp<128, 8>);
    }
    if (ce != cudaSuccess) return KVSEL_ERR_CUDA;
    if ((st = launch_status()) != KVSEL_OK) return st;
  } else {
    TraceScope ts("attend_split", s);
    if (d.head_dim == 64) {
      if (set_smem((const void*)attend_split<64>, smem) != cudaSuccess) return KVSEL_ERR_CUDA;
      attend_split<64><<<(unsigned)(rows * S), kAttThreads, smem, s>>>(a, t);
    } else {
      if (set_smem((const void*)attend_split<128>, smem) != cudaSuccess) return KVSEL_ERR_CUDA;
      attend_split<128><<<(unsigned)(rows * S), kAttThreads, smem, s>>>(a, t);
    }
    if ((st = launch_status()) != KVSEL_OK) return st;
  }
  TraceScope ts("attend_combine", s);
  if (d.head_dim == 64) attend_combine<64><<<(unsigned)(rows * a.R), 64, 0, s>>>(a);
  else attend_combine<128><<<(unsigned)(rows * a.R), 128, 0, s>>>(a);
  return launch_status();
}

}  // namespace kvsel
