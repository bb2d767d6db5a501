// Causal prefill attention on the 5th-generation tensor cores, emitting the window rows' log-sum-exp
// and queries for the scoring pass.
//
// CLAA, 'Complete flow and cost' (engineering detail 1): the keys that score the observation window
// are the prefill's own intermediate results.  The prefill's softmax already forms every row's
// log-sum-exp, which is exactly the first of the scoring's two passes over K for the window rows; so
// this kernel writes, besides o and the lse of every row, the window rows' lse (in the scoring's
// layout, base-2 units) and their queries, and the scoring then needs its second pass only.
//
// One CTA per (sequence, layer, query head, 128-row query tile), heaviest tiles first.  Warp 0
// issues TMA (the Q tile once; K and V tiles through a two-stage ring), warp 1 issues UMMA
// (S = Q K^T into one of two TMEM buffers; O += P V into a TMEM accumulator, V as an MN-major
// operand), warps 2..5 own one query row per thread: they read S from TMEM, apply the causal mask,
// keep the online (max, sum), write P as bf16 into shared memory in the swizzled K-major layout the
// UMMA reads, and rescale O in TMEM when a row's max grows.  All waits are bounded.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "internal.cuh"
#include "sm100.cuh"

namespace kvsel {
namespace {

using namespace sm100;

constexpr int kPfThreads = 192;
constexpr int kPfTile = 128;
constexpr uint32_t kQOff = 0, kPOff = 32768, kKVOff = 65536, kStageBytes = 65536;
constexpr uint32_t kBarOff = kKVOff + 2 * kStageBytes;               // 196608
// barriers: k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], s_empty[2], p_full, pv_done, q_full, drain
constexpr uint32_t kNumBars = 16;
constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
constexpr size_t kPfSmem = kMiscOff + 16 + 1024;
constexpr uint32_t kSCol = 0, kOCol = 256;                          // TMEM: S buffers 0..255, O 256..383

enum : uint32_t { kPfProducer = 11, kPfMma = 12, kPfSoftmax = 13, kPfDrain = 14 };

struct PfArgs {
  int32_t n_layers, h_q, h_kv, G, W, batch;
  float scale_log2;
  const __nv_bfloat16* q;       // full queries (window rows are copied from here)
  __nv_bfloat16* o;             // attention output, layout of q
  float* lse;                   // natural-log lse of every row (nullable)
  float* lse_win;               // base-2 lse of the window rows, [batch][layers][h_kv][G * W]
  __nv_bfloat16* q_win;         // window queries, [batch][layers][h_q][W][d]
  DeviceError* err;
  int32_t n_qt_max;
  int64_t q_row0[KVSEL_MAX_BATCH];   // first row of each sequence in the q / o row view
};

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool pf_aborted(const volatile uint32_t* f) { return *f != 0; }
__device__ __forceinline__ void pf_fail(const PfArgs& a, volatile uint32_t* f, uint32_t where) {
  set_device_error(a.err, KVSEL_ERR_TIMEOUT, where);
  *f = 1;
}

__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap tq,
                                                                const __grid_constant__ CUtensorMap tk,
                                                                const __grid_constant__ CUtensorMap tv,
                                                                const __grid_constant__ PfArgs a,
                                                                const __grid_constant__ SeqTable t) {
  constexpr int D = 128;
  const int heads_total = a.batch * a.n_layers * a.h_q;
  const int qt = a.n_qt_max - 1 - (int)(blockIdx.x / heads_total);   // heaviest tiles first
  const int hrem = (int)(blockIdx.x % heads_total);
  const int b = hrem / (a.n_layers * a.h_q);
  const int layer = (hrem / a.h_q) % a.n_layers;
  const int h = hrem % a.h_q;
  const int g = h / a.G;
  const SeqInfo& si = t.s[b];
  const int N = si.n_keys;
  if (qt * kPfTile >= N) return;                                      // this sequence is shorter
  const int nt = qt + 1;                                               // causal: K tiles 0 .. qt

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t base = smem_addr(sbase);
  const uint32_t bars = base + kBarOff;
  auto k_full = [&](int s) { return bars + 8u * s; };
  auto k_empty = [&](int s) { return bars + 8u * (2 + s); };
  auto v_full = [&](int s) { return bars + 8u * (4 + s); };
  auto v_empty = [&](int s) { return bars + 8u * (6 + s); };
  auto s_full = [&](int s) { return bars + 8u * (8 + s); };
  auto s_empty = [&](int s) { return bars + 8u * (10 + s); };
  const uint32_t p_full = bars + 96, pv_done = bars + 104, q_full = bars + 112, drain = bars + 120;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sbase + kMiscOff);
  volatile uint32_t* flag = reinterpret_cast<volatile uint32_t*>(sbase + kMiscOff + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
      mbar_init(s_full(s), 1);
      mbar_init(s_empty(s), 4);           // one arrival per softmax warp
    }
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
    mbar_init(q_full, 1);
    mbar_init(drain, 1);
    *flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(smem_addr(tslot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  const int64_t qrow0 = a.q_row0[b] + ((int64_t)layer * a.h_q + h) * N + (int64_t)qt * kPfTile;
  const int64_t krow0 = si.k_off / D + ((int64_t)layer * a.h_kv + g) * N;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_expect_tx(q_full, 32768);
      tma_load_2d(base + kQOff, &tq, 0, (int32_t)qrow0, q_full);
      tma_load_2d(base + kQOff + 16384, &tq, 64, (int32_t)qrow0, q_full);
      // K tiles are freed by their S product, V tiles by their P V product: two rings, filled in
      // tile order (K_j, V_j, K_j+1, ...)
      int kfills = 0, vfills = 0;
      for (int j = 0; j < nt; ++j) {
        const int s = j & 1;
        const uint32_t st = base + kKVOff + s * kStageBytes;
        const int32_t kr = (int32_t)(krow0 + (int64_t)j * kPfTile);
        if (pf_aborted(flag) || !mbar_wait(k_empty(s), ((j >> 1) & 1) ^ 1)) { pf_fail(a, flag, kPfProducer); break; }
        mbar_expect_tx(k_full(s), 32768);
        tma_load_2d(st, &tk, 0, kr, k_full(s));
        tma_load_2d(st + 16384, &tk, 64, kr, k_full(s));
        ++kfills;
        if (pf_aborted(flag) || !mbar_wait(v_empty(s), ((j >> 1) & 1) ^ 1)) { pf_fail(a, flag, kPfProducer); break; }
        mbar_expect_tx(v_full(s), 32768);
        tma_load_2d(st + 32768, &tv, 0, kr, v_full(s));
        tma_load_2d(st + 49152, &tv, 64, kr, v_full(s));
        ++vfills;
      }
      // copies still in flight (only after an abort) land before the CTA exits
      for (int s = 0; s < 2; ++s) {
        if (kfills > s && !mbar_wait(k_full(s), (((kfills - s + 1) / 2) - 1) & 1))
          set_device_error(a.err, KVSEL_ERR_TIMEOUT, kPfDrain);
        if (vfills > s && !mbar_wait(v_full(s), (((vfills - s + 1) / 2) - 1) & 1))
          set_device_error(a.err, KVSEL_ERR_TIMEOUT, kPfDrain);
      }
      if (!mbar_wait(q_full, 0)) set_device_error(a.err, KVSEL_ERR_TIMEOUT, kPfDrain);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(128, 128);
      constexpr uint32_t idesc_o = umma_idesc_bf16(128, 128) | kUmmaBMajorMN;
      bool ok = mbar_wait(q_full, 0);
      bool issued = false;
      auto issue_s = [&](int j) -> bool {
        const int s = j & 1;
        if (pf_aborted(flag) || !mbar_wait(k_full(s), (j >> 1) & 1) || !mbar_wait(s_empty(s), ((j >> 1) & 1) ^ 1))
          return false;
        tc_fence_after();
        const uint32_t sk = base + kKVOff + s * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t kb = kk >> 2, off = (kk & 3) * 32;
          umma_bf16(tmem + kSCol + s * 128, umma_desc_sw128(base + kQOff + kb * 16384 + off),
                    umma_desc_sw128(sk + kb * 16384 + off), idesc_s, kk > 0);
        }
        umma_commit(s_full(s));
        umma_commit(k_empty(s));
        issued = true;
        return true;
      };
      // S for the next two tiles is always in flight; the P V product of tile j comes first once its
      // P is ready, then S of tile j + 2 (whose K tile was loading meanwhile)
      if (ok) ok = issue_s(0);
      if (ok && nt > 1) ok = issue_s(1);
      for (int j = 0; j < nt && ok; ++j) {
        if (pf_aborted(flag) || !mbar_wait(p_full, j & 1) || !mbar_wait(v_full(j & 1), (j >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sv = base + kKVOff + (j & 1) * kStageBytes + 32768;
#pragma unroll
        for (int kk = 0; kk < kPfTile / 16; ++kk) {
          const uint32_t kb = kk >> 2, off = (kk & 3) * 32;
          umma_bf16(tmem + kOCol, umma_desc_sw128(base + kPOff + kb * 16384 + off),
                    umma_desc_sw128_mn(sv + kk * 2048, 16384), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(v_empty(j & 1));
        umma_commit(pv_done);
        if (j + 2 < nt && !issue_s(j + 2)) { ok = false; break; }
      }
      if (!ok) pf_fail(a, flag, kPfMma);
      if (issued) {
        umma_commit(drain);
        if (!mbar_wait(drain, 0)) set_device_error(a.err, KVSEL_ERR_TIMEOUT, kPfDrain);
      }
    }
  } else {
    // softmax / epilogue: thread = query row of the tile
    const int quarter = warp % 4;
    const int row = quarter * 32 + lane;
    const int i = qt * kPfTile + row;                               // row index in the sequence
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const float scale = a.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int s = j & 1;
      ok = __all_sync(0xffffffffu, ok && !pf_aborted(flag) && mbar_wait(s_full(s), (j >> 1) & 1));
      if (!ok) {
        if (lane == 0) pf_fail(a, flag, kPfSoftmax);
        break;
      }
      tc_fence_after();
      float v[128];
      tmem_ld64(lane_base + kSCol + s * 128, v);
      tmem_ld64(lane_base + kSCol + s * 128 + 64, v + 64);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty(s));
      // scale; causal mask on the diagonal tile (key j * 128 + c is visible to row i when c < i - 128 j + 1)
      if (j == nt - 1) {
        const int vis = i - j * kPfTile + 1;
#pragma unroll
        for (int c = 0; c < 128; ++c) v[c] = c < vis ? v[c] * scale : -INFINITY;
      } else {
#pragma unroll
        for (int c = 0; c < 128; ++c) v[c] *= scale;
      }
      float mp[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mp[k] = v[k];
#pragma unroll
      for (int c = 8; c < 128; ++c) mp[c & 7] = fmaxf(mp[c & 7], v[c]);
      const float mt = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])), fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      // lazy rescale: the exponent offset m moves only when the tile's max exceeds it by more than
      // 2^8, so O is rescaled in TMEM rarely (the probabilities stay below 256; the lse is m + log2 l
      // whatever m is)
      float alpha = 1.f;
      if (mt > m + 8.f) {
        alpha = m == -INFINITY ? 0.f : fast_ex2(m - mt);
        m = mt;
      }
      float sp[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) sp[k] = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = fast_ex2(v[2 * c] - m);
        const float p1 = fast_ex2(v[2 * c + 1] - m);
        sp[c & 7] += p0 + p1;
        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
        pk[c] = *reinterpret_cast<const uint32_t*>(&pb);
      }
      const float sum = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
      l = l * alpha + sum;
      // P and O may be touched once the previous tile's P V product is done
      if (j > 0) {
        ok = __all_sync(0xffffffffu, !pf_aborted(flag) && mbar_wait(pv_done, (j - 1) & 1));
        if (!ok) {
          if (lane == 0) pf_fail(a, flag, kPfSoftmax);
          break;
        }
        tc_fence_after();
      }
      // P row into the swizzled K-major tile: 64-key block kb at +16 KB, 16-byte chunk c at c ^ (row & 7)
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int kb = c >> 3, cc = c & 7;
        uint4 w = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        *reinterpret_cast<uint4*>(sbase + kPOff + kb * 16384 + row * 128 + ((cc ^ (row & 7)) * 16)) = w;
      }
      // rescale the running O when this row's max grew (warp-wide decision: the TMEM access is collective)
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        uint32_t r[64];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          tmem_ld64_async(lane_base + kOCol + half * 64, r);
          tmem_wait_ld64(r);
#pragma unroll
          for (int c = 0; c < 64; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
          tmem_st64(lane_base + kOCol + half * 64, r);
        }
        tmem_wait_st();
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, !pf_aborted(flag) && mbar_wait(pv_done, (nt - 1) & 1));
      if (!ok && lane == 0) pf_fail(a, flag, kPfSoftmax);
    }
    if (ok) {
      tc_fence_after();
      uint32_t r[64];
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool live = i < N;
      __nv_bfloat16* orow = a.o + (qrow0 + row) * D;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        tmem_ld64_async(lane_base + kOCol + half * 64, r);
        tmem_wait_ld64(r);
        if (live) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 pb = __floats2bfloat162_rn(__uint_as_float(r[8 * c + 2 * e]) * inv_l,
                                                              __uint_as_float(r[8 * c + 2 * e + 1]) * inv_l);
              w[e] = *reinterpret_cast<const uint32_t*>(&pb);
            }
            *reinterpret_cast<uint4*>(orow + half * 64 + c * 8) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (live) {
        const float lse2 = m + log2f(l);
        if (a.lse != nullptr) a.lse[qrow0 + row] = lse2 * 0.6931471805599453f;
        if (i >= si.L) {                                            // an observation-window row
          const int jw = i - si.L, hl = h - g * a.G;
          const int64_t unit = ((int64_t)b * a.n_layers + layer) * a.h_kv + g;
          a.lse_win[unit * (a.G * a.W) + hl * a.W + jw] = lse2;
          const uint4* src = reinterpret_cast<const uint4*>(a.q + (qrow0 + row) * D);
          uint4* dst = reinterpret_cast<uint4*>(a.q_win + ((((int64_t)b * a.n_layers + layer) * a.h_q + h) * a.W + jw) * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) dst[c] = src[c];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 pf_encode() {
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

bool pf_map(CUtensorMap* m, const void* ptr, int64_t rows) {
  auto fn = pf_encode();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

kvsel_status launch_prefill(const kvsel_desc& d, const SeqTable& t, const void* q, const void* k, const void* v,
                            void* o, float* lse, float* lse_win, void* q_win, DeviceError* err, cudaStream_t s) {
  PfArgs a;
  memset(&a, 0, sizeof(a));
  a.n_layers = d.n_layers;
  a.h_q = d.h_q;
  a.h_kv = d.h_kv;
  a.G = d.h_q / d.h_kv;
  a.W = d.window;
  a.batch = d.batch;
  a.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)d.head_dim));
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.lse_win = lse_win;
  a.q_win = static_cast<__nv_bfloat16*>(q_win);
  a.err = err;
  int64_t q_rows = 0, k_rows = 0, nmax = 0;
  for (int b = 0; b < d.batch; ++b) {
    a.q_row0[b] = q_rows;
    const int64_t n = t.s[b].n_keys;
    q_rows += (int64_t)d.n_layers * d.h_q * n;
    k_rows += (int64_t)d.n_layers * d.h_kv * n;
    nmax = n > nmax ? n : nmax;
  }
  if (q_rows + kPfTile >= (int64_t(1) << 31) || k_rows + kPfTile >= (int64_t(1) << 31)) return KVSEL_ERR_UNSUPPORTED;
  a.n_qt_max = (int32_t)((nmax + kPfTile - 1) / kPfTile);
  CUtensorMap tq, tk, tv;
  if (!pf_map(&tq, q, q_rows) || !pf_map(&tk, k, k_rows) || !pf_map(&tv, v, k_rows)) return KVSEL_ERR_CUDA;
  if (set_smem((const void*)prefill_kernel, kPfSmem) != cudaSuccess) return KVSEL_ERR_CUDA;
  const int64_t grid = (int64_t)a.n_qt_max * d.batch * d.n_layers * d.h_q;
  if (grid >= (int64_t(1) << 31)) return KVSEL_ERR_UNSUPPORTED;
  TraceScope ts("prefill_tc", s);
  prefill_kernel<<<(unsigned)grid, kPfThreads, kPfSmem, s>>>(tq, tk, tv, a, t);
  return launch_status();
}

}  // namespace kvsel
