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
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "sm100.cuh"

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
  int32_t rows;               // table rows (batch x layers x KV heads)
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
                                                            const __grid_constant__ SeqTable tp) {
  const SeqTable& t = real_table(tp);
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
  const SeqInfo si = t.s[b];   // a copy: loads once, whatever the table lives in
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
// step's K and V rows into one of the warp's three shared-memory stages with cp.async (whole rows per
// copy instruction; zero-filled where a position selects no row; 16-byte chunks XOR-swizzled by the
// key so that the matrix loads below hit distinct banks), two steps ahead of the step computed.  The arithmetic runs on mma.sync m16n8k16 (bf16 in, fp32 accumulate) with the
// group's query rows as the 16 rows of the A operand (rows R..15 zero): the logits S = Q K^T with Q
// held in registers for the whole split and K loaded by ldmatrix (bf16 products are exact, so this is
// the fp32 dot product up to summation order); P is formed in the logits' accumulator layout, which is
// the A-operand layout of the next product, and split into bf16 high and low parts so that P V is
// taken to ~16 significant bits of P; V is loaded transposed by ldmatrix.  The online softmax keeps an
// exponent offset that moves only when a row's max passes it by 2^8 (then O and l are rescaled).
// Warp w of the grid takes split w % S of table row w / S (the warps of one CTA may serve different
// rows), so the split count can be sized to fill exactly one wave of resident warps.
constexpr int kWarpsPerCta = 4;
constexpr int kStep = 16;
constexpr int kStages = 3;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const uint32_t n = valid ? 16u : 0u;   // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += A B for one 16x8x16 tile whose A rows 8..15 are zero (a1 = a3 = 0): only the accumulator
// elements of rows 0..7 (d[0], d[1]: row gq, columns 2tq and 2tq + 1) are kept.
__device__ __forceinline__ void mma_rows8(float* d, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  float x2, x3;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %10, %10};"
      : "+f"(d[0]), "+f"(d[1]), "=f"(x2), "=f"(x3)
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.f));
  asm volatile("" ::"f"(x2), "f"(x3));   // (rows 8..15 of the product: zero, unused)
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

template <int D>
__global__ void __launch_bounds__(32 * kWarpsPerCta) attend_warp(const __grid_constant__ AttArgs a,
                                                                 const __grid_constant__ SeqTable tp) {
  const SeqTable& t = real_table(tp);
  constexpr int VPR = D / 8;          // 16-byte chunks per row
  constexpr int STAGE = kStep * D;    // bf16 elements of one K (or V) stage
  constexpr int NT = D / 8;           // 8-wide tiles of the head dim in O
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;                           // fragment row / column pair
  __nv_bfloat16* Kb = reinterpret_cast<__nv_bfloat16*>(smem_raw) + warp * 2 * kStages * STAGE;   // [3][16][D]
  __nv_bfloat16* Vb = Kb + kStages * STAGE;                                                     // [3][16][D]
  const int64_t w = (int64_t)blockIdx.x * kWarpsPerCta + warp;
  if (w >= (int64_t)a.rows * a.S) return;                            // past the last split (whole warp)
  const int r = (int)(w / a.S);
  const int s = (int)(w % a.S);
  const int per_seq = a.n_layers * a.h_kv;
  const int b = r / per_seq, lg = r % per_seq;
  const int layer = lg / a.h_kv, g = lg % a.h_kv;
  const SeqInfo si = t.s[b];   // a copy: loads once, whatever the table lives in
  // A fragments of query row gq (zero for gq >= R): elements 16c + 2tq, +1 and 16c + 8 + 2tq, +1
  uint32_t qa[D / 16][2];
  {
    const bool live = gq < a.R;
    const int h = g * a.G + gq / a.n_q, i = gq % a.n_q;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        a.q + (live ? ((((int64_t)b * a.n_layers + layer) * a.h_q + h) * a.n_q + i) * D : 0));
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      qa[c][0] = live ? __ldg(qrow + 8 * c + tq) : 0u;
      qa[c][1] = live ? __ldg(qrow + 8 * c + 4 + tq) : 0u;
    }
  }
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
      const uint32_t dst = (uint32_t)((buf * STAGE + x * D) * 2 + ((c ^ (x & (VPR - 1))) * 16));
      cp_async16(kb_s + dst, kbase + src, rx >= 0);
      cp_async16(vb_s + dst, vbase + src, rx >= 0);
    }
    cp_async_commit();
  };
  // ldmatrix row addresses of this lane within a stage (byte offsets, before the chunk swizzle):
  // K: matrices (keys 0-7 | 8-15) x (low | high 8 of a 16-wide chunk); V (transposed): matrices
  // (keys 0-7 | 8-15) x (d tile 2p | 2p + 1)
  const int key_k = ((lane >> 4) << 3) | (lane & 7), hi_k = (lane >> 3) & 1;
  const int key_v = (((lane >> 3) & 1) << 3) | (lane & 7), hi_v = lane >> 4;

  float o[NT][2];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = 0.f;
  float m = -INFINITY, l = 0.f;
  const float scale = a.scale_log2;
  // every step commits one copy group (empty past the split's end), so waiting for all but the two
  // newest groups waits for exactly the step about to be computed
  int32_t row = row_of(p0 + key, id_at(p0 + key));
  if (p0 < p1) issue(row, 0); else cp_async_commit();
  int32_t row1 = row_of(p0 + kStep + key, id_at(p0 + kStep + key));
  if (p0 + kStep < p1) issue(row1, 1); else cp_async_commit();
  int32_t id_next = id_at(p0 + 2 * kStep + key);
  int buf = 0;
  for (int64_t base = p0; base < p1; base += kStep) {
    int32_t row2 = -1;
    const int32_t id_after = id_at(base + 3 * kStep + key);
    if (base + 2 * kStep < p1) {
      row2 = row_of(base + 2 * kStep + key, id_next);
      issue(row2, buf == 0 ? 2 : buf - 1);
    } else {
      cp_async_commit();
    }
    cp_async_wait<2>();
    id_next = id_after;
    __syncwarp();
    // logits of row gq: keys 2tq, 2tq + 1 (s0[0..1]) and 8 + 2tq, 9 + 2tq (s1[0..1])
    const uint32_t kst = kb_s + (uint32_t)(buf * STAGE * 2), vst = vb_s + (uint32_t)(buf * STAGE * 2);
    float s0[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f};
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      uint32_t kb[4];
      ldsm_x4(kb, kst + (uint32_t)(key_k * D * 2 + (((2 * c + hi_k) ^ (key_k & (VPR - 1))) << 4)));
      mma_rows8(s0, qa[c][0], qa[c][1], kb[0], kb[1]);
      mma_rows8(s1, qa[c][0], qa[c][1], kb[2], kb[3]);
    }
    const uint32_t valid = __ballot_sync(0xffffffffu, row >= 0);    // bit x: key x selects a row
    const int k0 = 2 * tq;
    float z[4] = {s0[0], s0[1], s1[0], s1[1]};
    const int kz[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
#pragma unroll
    for (int e = 0; e < 4; ++e) z[e] = ((valid >> kz[e]) & 1u) ? z[e] * scale : -INFINITY;
    float mx = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    float alpha = 1.f;
    if (mx > m + 8.f) {
      alpha = m == -INFINITY ? 0.f : fast_ex2(m - mx);
      m = mx;
    }
    if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][0] *= alpha;
        o[n][1] *= alpha;
      }
    }
    float p[4], sum = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      p[e] = z[e] == -INFINITY ? 0.f : fast_ex2(z[e] - m);
      sum += p[e];
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    l = l * alpha + sum;
    // P as bf16 high + low parts, in the A-operand layout (keys 2tq.. in a0, 8 + 2tq.. in a2)
    const uint32_t h01 = pack_bf16(p[0], p[1]), h23 = pack_bf16(p[2], p[3]);
    const __nv_bfloat162 hb01 = *reinterpret_cast<const __nv_bfloat162*>(&h01);
    const __nv_bfloat162 hb23 = *reinterpret_cast<const __nv_bfloat162*>(&h23);
    const uint32_t l01 = pack_bf16(p[0] - __low2float(hb01), p[1] - __high2float(hb01));
    const uint32_t l23 = pack_bf16(p[2] - __low2float(hb23), p[3] - __high2float(hb23));
#pragma unroll
    for (int pp = 0; pp < NT / 2; ++pp) {
      uint32_t vb[4];
      ldsm_x4_t(vb, vst + (uint32_t)(key_v * D * 2 + (((2 * pp + hi_v) ^ (key_v & (VPR - 1))) << 4)));
      mma_rows8(o[2 * pp], h01, h23, vb[0], vb[1]);
      mma_rows8(o[2 * pp], l01, l23, vb[0], vb[1]);
      mma_rows8(o[2 * pp + 1], h01, h23, vb[2], vb[3]);
      mma_rows8(o[2 * pp + 1], l01, l23, vb[2], vb[3]);
    }
    __syncwarp();          // the stage is read before it is refilled
    row = row1;
    row1 = row2;
    buf = buf == kStages - 1 ? 0 : buf + 1;
  }
  cp_async_wait<0>();      // (only empty groups can remain)
  if (gq < a.R) {
    float* out = a.part + (((int64_t)r * a.S + s) * a.R + gq) * (D + 2);
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      out[8 * n + 2 * tq] = o[n][0];
      out[8 * n + 2 * tq + 1] = o[n][1];
    }
    if (tq == 0) {
      out[D] = m;
      out[D + 1] = l;
    }
  }
}

size_t attend_warp_smem(int d) { return (size_t)kWarpsPerCta * 2 * kStages * kStep * d * 2; }

// ---------------------------------------------------------------- the same warp kernel, stages by TMA
// When the 16 rows of every step are consecutive cache rows (whole caches, or blocks of a multiple of
// 16 rows), each step's K and V rows are one 16-row box of a 2-D tensor map over the cache ([rows][d],
// 64-column boxes with the 128-byte swizzle): one lane issues the step's box loads, which complete on
// the stage's mbarrier, instead of 32 lanes issuing 16-byte copies, and the block ids are loaded a
// step before their loads are issued.  The arithmetic is the warp kernel's (two accumulation chains
// per logit tile); K and V are addressed in the swizzled layout (16-byte chunk c of row x of a
// 64-column half at (c ^ (x & 7)) * 16).
constexpr uint32_t kHalfBytes = kStep * 128;   // one 64-column half of a stage's 16 rows
constexpr int kTmaStages = 3;   // stages per warp: two steps in flight
constexpr int kTmaWarps = 4;    // warps per CTA (two CTAs of 4 x 24 KB per SM at d = 128)

template <int D>
__host__ __device__ constexpr uint32_t tma_stage_bytes() { return (uint32_t)(D / 64) * kHalfBytes; }   // K (or V) of one stage

size_t attend_tma_smem(int d) {
  const size_t stages = (size_t)kTmaWarps * 2 * kTmaStages * (d / 64) * kHalfBytes;
  return 1024 + stages + (size_t)kTmaWarps * kTmaStages * 12;   // slack, stages, mbarriers and step rows
}

template <int D>
__global__ void __launch_bounds__(32 * kTmaWarps) attend_tma(const __grid_constant__ CUtensorMap tmk,
                                                                const __grid_constant__ CUtensorMap tmv,
                                                                const __grid_constant__ AttArgs a,
                                                                const __grid_constant__ SeqTable tp) {
  const SeqTable& t = real_table(tp);
  constexpr int NT = D / 8;
  constexpr uint32_t KV = tma_stage_bytes<D>();
  constexpr int NS = kTmaStages;
  constexpr uint32_t WARP_BYTES = 2 * NS * KV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const uint32_t st0 = sm100::smem_addr(sbase) + warp * WARP_BYTES;          // K stages, then V stages
  const uint32_t bar0 = sm100::smem_addr(sbase) + kTmaWarps * WARP_BYTES + warp * NS * 8;
  // first cache row of the step in each stage (written by the issuing lane)
  volatile int32_t* rows_s = reinterpret_cast<volatile int32_t*>(sbase + kTmaWarps * (WARP_BYTES + NS * 8)) + warp * NS;
  const int64_t w = (int64_t)blockIdx.x * kTmaWarps + warp;
  if (w >= (int64_t)a.rows * a.S) return;                                    // whole warp
  if (lane == 0) {
    for (int i = 0; i < NS; ++i) sm100::mbar_init(bar0 + 8u * i, 1);
    sm100::fence_barrier_init();
  }
  __syncwarp();
  const int r = (int)(w / a.S);
  const int s = (int)(w % a.S);
  const int per_seq = a.n_layers * a.h_kv;
  const int b = r / per_seq, lg = r % per_seq;
  const int layer = lg / a.h_kv, g = lg % a.h_kv;
  const SeqInfo si = t.s[b];
  uint32_t qa[D / 16][2];
  {
    const bool live = gq < a.R;
    const int h = g * a.G + gq / a.n_q, i = gq % a.n_q;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        a.q + (live ? ((((int64_t)b * a.n_layers + layer) * a.h_q + h) * a.n_q + i) * D : 0));
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      qa[c][0] = live ? __ldg(qrow + 8 * c + tq) : 0u;
      qa[c][1] = live ? __ldg(qrow + 8 * c + 4 + tq) : 0u;
    }
  }
  int beg, end;
  row_list(a, si, r, beg, end);
  // positions of the row in steps of 16 (blocks hold whole steps); this split's steps
  const int64_t n_pos = (int64_t)(end - beg) * a.P;
  const int64_t n_steps = (n_pos + kStep - 1) / kStep;
  const int64_t p0 = ((s * n_steps) / a.S) * kStep;
  const int64_t p1 = min(n_pos, (((s + 1) * n_steps) / a.S) * kStep);
  const int32_t unit_row0 = (int32_t)(si.k_off / D + ((int64_t)layer * a.h_kv + g) * si.n_keys);
  const int key = lane & (kStep - 1);

  // Block id of the step at `pos` (loaded a step before it is needed), then the step's first cache
  // row, or -1 (past the split, or a block outside the cache).
  auto step_id = [&](int64_t pos) -> int32_t {
    if (pos >= p1) return -1;
    const int bi = (int)(pos / a.P);
    return a.indices == nullptr ? bi : __ldg(a.indices + beg + bi);
  };
  auto step_row = [&](int64_t pos, int32_t id) -> int32_t {
    if (pos >= p1) return -1;
    const int bi = (int)(pos / a.P), within = (int)(pos - (int64_t)bi * a.P);
    const int64_t rr = (int64_t)id * a.P + within;
    if (id >= 0 && rr < si.n_keys) return (int32_t)rr;
    if (within == 0 && lane == 0) set_device_error(a.err, KVSEL_ERR_DEVICE, (uint32_t)(beg + bi));
    return -1;
  };
  // One lane loads the step's K and V boxes into stage `buf` (a step with no row loads row 0 of the
  // unit: its keys are masked).
  auto issue = [&](int32_t row0, int buf) {
    if (lane == 0) {
      rows_s[buf] = row0;
      const uint32_t bar = bar0 + 8u * buf;
      sm100::mbar_expect_tx(bar, 2 * KV);
      const int32_t y = unit_row0 + (row0 < 0 ? 0 : row0);
      const uint32_t kst = st0 + buf * KV, vst = st0 + NS * KV + buf * KV;
#pragma unroll
      for (int hh = 0; hh < D / 64; ++hh) {
        sm100::tma_load_2d(kst + hh * kHalfBytes, &tmk, 64 * hh, y, bar);
        sm100::tma_load_2d(vst + hh * kHalfBytes, &tmv, 64 * hh, y, bar);
      }
    }
  };
  // swizzled byte offset of 16-byte chunk cc (0 .. D/8 - 1) of row x within a K or V stage
  auto chunk_at = [](int x, int cc) -> uint32_t {
    return (uint32_t)((cc >> 3) * kHalfBytes + x * 128 + (((cc & 7) ^ (x & 7)) << 4));
  };
  const int key_k = ((lane >> 4) << 3) | (lane & 7), hi_k = (lane >> 3) & 1;
  const int key_v = (((lane >> 3) & 1) << 3) | (lane & 7), hi_v = lane >> 4;

  float o[NT][2];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = 0.f;
  float m = -INFINITY, l = 0.f;
  const float scale = a.scale_log2;
  // steps are issued NS - 1 ahead; step k uses stage k % NS with phase (k / NS) & 1
#pragma unroll
  for (int i = 0; i < NS - 1; ++i) {
    const int64_t pos = p0 + (int64_t)i * kStep;
    if (pos < p1) issue(step_row(pos, step_id(pos)), i);
  }
  int32_t id_c = step_id(p0 + (int64_t)(NS - 1) * kStep);          // block of the next step to issue
  int64_t k_step = 0;
  bool ok = true;
  for (int64_t base = p0; base < p1; base += kStep, ++k_step) {
    const int buf = (int)(k_step % NS);
    const int64_t npos = base + (int64_t)(NS - 1) * kStep;
    const int32_t id_d = step_id(npos + kStep);                    // used at the next step
    if (npos < p1) {
      const int32_t row_c = step_row(npos, id_c);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the stage's last reads come first
      issue(row_c, (int)((k_step + NS - 1) % NS));
    }
    id_c = id_d;
    const uint32_t parity = (uint32_t)((k_step / NS) & 1);
    if (!__all_sync(0xffffffffu, sm100::mbar_wait(bar0 + 8u * buf, parity))) {
      if (lane == 0) set_device_error(a.err, KVSEL_ERR_TIMEOUT, 5u);
      ok = false;
      break;
    }
    const int32_t row0 = rows_s[buf];
    const uint32_t kst = st0 + buf * KV, vst = st0 + NS * KV + buf * KV;
    // two accumulation chains per 8-key tile (even / odd 16-wide chunks of d), added at the end
    float s0[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f}, t0[2] = {0.f, 0.f}, t1[2] = {0.f, 0.f};
#pragma unroll
    for (int c = 0; c < D / 16; c += 2) {
      uint32_t kb[4], kc[4];
      ldsm_x4(kb, kst + chunk_at(key_k, 2 * c + hi_k));
      ldsm_x4(kc, kst + chunk_at(key_k, 2 * c + 2 + hi_k));
      mma_rows8(s0, qa[c][0], qa[c][1], kb[0], kb[1]);
      mma_rows8(s1, qa[c][0], qa[c][1], kb[2], kb[3]);
      mma_rows8(t0, qa[c + 1][0], qa[c + 1][1], kc[0], kc[1]);
      mma_rows8(t1, qa[c + 1][0], qa[c + 1][1], kc[2], kc[3]);
    }
    s0[0] += t0[0];
    s0[1] += t0[1];
    s1[0] += t1[0];
    s1[1] += t1[1];
    // key x of the step is row row0 + x: it exists when the step has a row, the position lies in the
    // split and the row lies in the cache (a block may end past the cache)
    const bool kv_ok = row0 >= 0 && base + key < p1 && row0 + key < si.n_keys;
    const uint32_t valid = __ballot_sync(0xffffffffu, kv_ok && lane < kStep);
    const int k0 = 2 * tq;
    float z[4] = {s0[0], s0[1], s1[0], s1[1]};
    const int kz[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
#pragma unroll
    for (int e = 0; e < 4; ++e) z[e] = ((valid >> kz[e]) & 1u) ? z[e] * scale : -INFINITY;
    float mx = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    float alpha = 1.f;
    if (mx > m + 8.f) {
      alpha = m == -INFINITY ? 0.f : fast_ex2(m - mx);
      m = mx;
    }
    if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][0] *= alpha;
        o[n][1] *= alpha;
      }
    }
    float p[4], sum = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      p[e] = z[e] == -INFINITY ? 0.f : fast_ex2(z[e] - m);
      sum += p[e];
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    l = l * alpha + sum;
    const uint32_t h01 = pack_bf16(p[0], p[1]), h23 = pack_bf16(p[2], p[3]);
    const __nv_bfloat162 hb01 = *reinterpret_cast<const __nv_bfloat162*>(&h01);
    const __nv_bfloat162 hb23 = *reinterpret_cast<const __nv_bfloat162*>(&h23);
    const uint32_t l01 = pack_bf16(p[0] - __low2float(hb01), p[1] - __high2float(hb01));
    const uint32_t l23 = pack_bf16(p[2] - __low2float(hb23), p[3] - __high2float(hb23));
#pragma unroll
    for (int pp = 0; pp < NT / 2; ++pp) {
      uint32_t vb[4];
      ldsm_x4_t(vb, vst + chunk_at(key_v, 2 * pp + hi_v));
      mma_rows8(o[2 * pp], h01, h23, vb[0], vb[1]);
      mma_rows8(o[2 * pp], l01, l23, vb[0], vb[1]);
      mma_rows8(o[2 * pp + 1], h01, h23, vb[2], vb[3]);
      mma_rows8(o[2 * pp + 1], l01, l23, vb[2], vb[3]);
    }
    __syncwarp();          // every lane's reads of the stage precede its next load
  }
  if (!ok) {
    // loads still in flight must land before the warp exits: wait (bounded) for every issued step
    for (int64_t k2 = k_step; k2 < k_step + NS - 1; ++k2) {
      if (p0 + k2 * kStep >= p1) break;
      sm100::mbar_wait(bar0 + 8u * (uint32_t)(k2 % NS), (uint32_t)((k2 / NS) & 1));
    }
    return;
  }
  if (gq < a.R) {
    float* out = a.part + (((int64_t)r * a.S + s) * a.R + gq) * (D + 2);
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      out[8 * n + 2 * tq] = o[n][0];
      out[8 * n + 2 * tq + 1] = o[n][1];
    }
    if (tq == 0) {
      out[D] = m;
      out[D + 1] = l;
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 att_encode() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D view [rows][d] bf16 of a cache, boxes of 64 columns x 16 rows with the 128-byte swizzle.
bool att_map(CUtensorMap* mp, const void* ptr, int64_t rows, int d) {
  auto fn = att_encode();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kStep};
  cuuint32_t es[2] = {1, 1};
  return fn(mp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

using AttKernel = void (*)(const AttArgs, const SeqTable);

// The warp kernel for head dim d (any R <= 8 query rows per table row).
AttKernel attend_warp_kernel(int d) { return d == 64 ? attend_warp<64> : attend_warp<128>; }

// Warps of the warp kernel resident at once on the current device; 0 if that cannot be queried.
// Queried once per (device, head dim).
int64_t attend_resident_warps(int d) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static int64_t cache[kMaxDev][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int di = d == 64 ? 0 : 1;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < kMaxDev && cache[dev][di] > 0) return cache[dev][di];
  const size_t wsm = attend_warp_smem(d);
  const AttKernel kern = attend_warp_kernel(d);
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      set_smem((const void*)kern, wsm) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * kWarpsPerCta, wsm) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int64_t n = (int64_t)sms * per_sm * kWarpsPerCta;
  if (dev >= 0 && dev < kMaxDev) cache[dev][di] = n;
  return n;
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

// Warps of the TMA warp kernel resident at once on the current device (0 if that cannot be queried).
int64_t attend_tma_resident_warps(int d) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static int64_t cache[kMaxDev][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int di = d == 64 ? 0 : 1;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < kMaxDev && cache[dev][di] > 0) return cache[dev][di];
  const size_t wsm = attend_tma_smem(d);
  const void* kern = d == 64 ? (const void*)attend_tma<64> : (const void*)attend_tma<128>;
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      set_smem(kern, wsm) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * kTmaWarps, wsm) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int64_t n = (int64_t)sms * per_sm * kTmaWarps;
  if (dev >= 0 && dev < kMaxDev) cache[dev][di] = n;
  return n;
}

int64_t attend_splits(int64_t rows, int64_t max_rows_per_list, int R, int d, int block) {
  if (R <= 8) {
    // warp splits: as many as fit one wave of resident warps (all rows' splits run at once), no
    // split shorter than 64 positions.  Blocks of a multiple of 16 rows run on the TMA kernel.
    int64_t resident = block % kStep == 0 ? attend_tma_resident_warps(d) : attend_resident_warps(d);
    if (resident <= 0) resident = 152 * 12;
    int64_t s = resident / rows;
    const int64_t cap = (max_rows_per_list + 63) / 64;
    if (s > cap) s = cap;
    if (s < 1) s = 1;
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
  a.rows = (int32_t)rows;
  const size_t smem = attend_smem(d.head_dim);
  kvsel_status st;
  // every step's 16 rows consecutive: whole caches, or blocks of a multiple of 16 rows
  int64_t cache_rows = 0;
  for (int b = 0; b < d.batch; ++b) cache_rows += (int64_t)d.n_layers * d.h_kv * t.s[b].n_keys;
  CUtensorMap tmk, tmv;
  const bool tma = a.R <= 8 && (indices == nullptr || P % kStep == 0) && cache_rows + kStep < (int64_t(1) << 31) &&
                   att_map(&tmk, k, cache_rows, d.head_dim) && att_map(&tmv, v, cache_rows, d.head_dim);
  if (tma) {
    TraceScope ts("attend_split", s);
    const unsigned grid = (unsigned)((rows * S + kTmaWarps - 1) / kTmaWarps);
    const size_t wsm = attend_tma_smem(d.head_dim);
    if (d.head_dim == 64) {
      if (set_smem((const void*)attend_tma<64>, wsm) != cudaSuccess) return KVSEL_ERR_CUDA;
      attend_tma<64><<<grid, 32 * kTmaWarps, wsm, s>>>(tmk, tmv, a, t);
    } else {
      if (set_smem((const void*)attend_tma<128>, wsm) != cudaSuccess) return KVSEL_ERR_CUDA;
      attend_tma<128><<<grid, 32 * kTmaWarps, wsm, s>>>(tmk, tmv, a, t);
    }
    if ((st = launch_status()) != KVSEL_OK) return st;
  } else if (a.R <= 8) {
    TraceScope ts("attend_split", s);
    const unsigned grid = (unsigned)((rows * S + kWarpsPerCta - 1) / kWarpsPerCta);
    const size_t wsm = attend_warp_smem(d.head_dim);
    const AttKernel kern = attend_warp_kernel(d.head_dim);
    if (set_smem((const void*)kern, wsm) != cudaSuccess) return KVSEL_ERR_CUDA;
    kern<<<grid, 32 * kWarpsPerCta, wsm, s>>>(a, t);
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
