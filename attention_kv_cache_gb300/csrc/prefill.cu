// Causal prefill attention on the 5th-generation tensor cores, emitting the window rows' log-sum-exp
// and queries for the scoring pass.
//
// CLAA, 'Complete flow and cost' (engineering detail 1): the keys that score the observation window
// are the prefill's own intermediate results.  The prefill's softmax already forms every row's
// log-sum-exp, which is exactly the first of the scoring's two passes over K for the window rows; so
// this kernel writes, besides o and the lse of every row, the window rows' lse (in the scoring's
// layout, base-2 units) and their queries, and the scoring then needs its second pass only.
//
// One CTA per (sequence, layer, query head, pair of consecutive 128-row query tiles A and B),
// heaviest pairs first.  The two tiles share every K and V tile; while one tile's softmax runs, the
// tensor cores work on the other's products.  Warp 0 issues TMA (both Q tiles once; K and V tiles
// through two-stage rings); warp 1 issues UMMA: S_X = Q_X K^T into TMEM, O_X += P_X V with P_X read
// from TMEM (written there over S_X by the softmax) and V as an MN-major shared-memory operand.
// The eight steps of one product form a dependent accumulation chain, which the tensor pipe runs
// well below its rate; two independent products issued step by step in alternation run near it.
// Tile B trails tile A by one S product, so that B's P V of step j becomes ready when A's P V of
// step j completes, i.e. when A's next S may start: those two are issued interleaved, and the
// order per step is P_A V, (P_B V | S_A of the next step), S_B of the next step.  Warps 2..5
// (tile A) and 6..9 (tile B) own one query row per thread: they read S from TMEM, apply the causal
// mask, keep an exponent offset that moves only past 2^8 (so O is rescaled in TMEM rarely), and
// store P as bf16 pairs.  A tile's next S is issued only after its P V product has completed, which
// orders every reuse of its TMEM columns.  All waits are bounded.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "internal.cuh"
#include "sm100.cuh"

namespace kvsel {
namespace {

using namespace sm100;

constexpr int kPfThreads = 320;
constexpr int kPfTile = 128;
// shared memory: Q_A | Q_B | K stages | V stages (32 KB each), then barriers
constexpr uint32_t kQOff = 0, kKOff = 65536, kVOff = 131072, kTileBytes = 32768;
constexpr uint32_t kBarOff = 196608;
// barriers: k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2], pv_done[2], q_full, drain
constexpr uint32_t kNumBars = 16;
constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
constexpr size_t kPfSmem = kMiscOff + 16 + 1024;
// TMEM: tile X in {0, 1}: S (P over its first 64 columns) at 256 X, O at 256 X + 128
constexpr uint32_t kSCol = 0, kOCol = 128, kTileCols = 256;

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
  int32_t n_pairs;              // query-tile pairs of the longest sequence
};

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool pf_aborted(const volatile uint32_t* f) { return *f != 0; }

// A wait on the pipeline's critical path: polls without sleeping, and reads the abort flag only every
// 256 polls (under the tensor pipe's and TMA's shared-memory traffic every shared-memory access of
// the polling thread costs on the order of a hundred cycles, so a phase that has completed must
// cost one access, not two).  False after kSpinLimit polls or once another role has aborted.
__device__ __forceinline__ bool pf_wait(uint32_t bar, uint32_t parity, const volatile uint32_t* f) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 255 && pf_aborted(f)) return false;
  }
  return false;
}
__device__ __forceinline__ void pf_fail(const PfArgs& a, volatile uint32_t* f, uint32_t where) {
  set_device_error(a.err, KVSEL_ERR_TIMEOUT, where);
  *f = 1;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Largest of 64 raw logits (three-input max: 36 instructions).
__device__ __forceinline__ float max64(const float* v) {
  float mp[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float* c = v + 8 * k;
    mp[k] = fmaxf(fmax3(fmax3(c[0], c[1], c[2]), c[3], c[4]), fmax3(c[5], c[6], c[7]));
  }
  return fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
}

// Causal mask of 64 raw logits of keys key0 .. key0 + 63 for row i: keys after i become -inf.
__device__ __forceinline__ void mask64(float* v, int key0, int i) {
  const int vis = i - key0 + 1;
#pragma unroll
  for (int c = 0; c < 64; ++c) v[c] = c < vis ? v[c] : -INFINITY;
}

// 2^(scale v - m) of 64 raw logits, two per packed fma: their sum, and the bf16 pairs in 32 words
// (even key in the low half).  pk may be v's own registers: word c is written after v[2c] and
// v[2c + 1] are read.
__device__ __forceinline__ float exp_pack64(const float* v, float2 sc, float2 nm, uint32_t* pk) {
  float2 sp[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) sp[k] = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const float2 t = __ffma2_rn(make_float2(v[2 * c], v[2 * c + 1]), sc, nm);
    const float2 p = make_float2(fast_ex2(t.x), fast_ex2(t.y));
    sp[c & 3] = __fadd2_rn(sp[c & 3], p);
    const __nv_bfloat162 pb = __floats2bfloat162_rn(p.x, p.y);
    pk[c] = *reinterpret_cast<const uint32_t*>(&pb);
  }
  const float2 s = __fadd2_rn(__fadd2_rn(sp[0], sp[1]), __fadd2_rn(sp[2], sp[3]));
  return s.x + s.y;
}

__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap tq,
                                                                const __grid_constant__ CUtensorMap tk,
                                                                const __grid_constant__ CUtensorMap tv,
                                                                const __grid_constant__ PfArgs a,
                                                                const __grid_constant__ SeqTable tp) {
  const SeqTable& t = real_table(tp);
  constexpr int D = 128;
  const int heads_total = a.batch * a.n_layers * a.h_q;
  const int pair = a.n_pairs - 1 - (int)(blockIdx.x / heads_total);   // heaviest pairs first
  const int hrem = (int)(blockIdx.x % heads_total);
  const int b = hrem / (a.n_layers * a.h_q);
  const int layer = (hrem / a.h_q) % a.n_layers;
  const int h = hrem % a.h_q;
  const int g = h / a.G;
  const SeqInfo si = t.s[b];   // a copy: loads once, whatever the table lives in
  const int N = si.n_keys;
  const int qa = 2 * pair;
  if (qa * kPfTile >= N) return;                                       // this sequence is shorter
  const int nq = (qa + 1) * kPfTile < N ? 2 : 1;                        // query tiles in this CTA
  const int nt_x[2] = {qa + 1, qa + 2};                                 // K tiles of tile A, B (causal)
  const int nt = nt_x[nq - 1];

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t base = smem_addr(sbase);
  const uint32_t bars = base + kBarOff;
  auto k_full = [&](int s) { return bars + 8u * s; };
  auto k_empty = [&](int s) { return bars + 8u * (2 + s); };
  auto v_full = [&](int s) { return bars + 8u * (4 + s); };
  auto v_empty = [&](int s) { return bars + 8u * (6 + s); };
  auto s_full = [&](int x) { return bars + 8u * (8 + x); };
  auto p_full = [&](int x) { return bars + 8u * (10 + x); };
  auto pv_done = [&](int x) { return bars + 8u * (12 + x); };
  const uint32_t q_full = bars + 112, drain = bars + 120;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sbase + kMiscOff);
  volatile uint32_t* flag = reinterpret_cast<volatile uint32_t*>(sbase + kMiscOff + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), nq);          // freed by the S product of every tile that reads it
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), nq);          // freed by the P V product of every tile that reads it
      mbar_init(s_full(s), 1);
      mbar_init(p_full(s), 4);            // one arrival per softmax warp of the tile
      mbar_init(pv_done(s), 1);
    }
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

  // the sequence's first q / o row: its K rows (k_off / d) times the G query heads per KV head
  const int64_t qrow_base = si.k_off / D * a.G + ((int64_t)layer * a.h_q + h) * N;
  const int64_t krow0 = si.k_off / D + ((int64_t)layer * a.h_kv + g) * N;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_expect_tx(q_full, 32768u * nq);
      for (int x = 0; x < nq; ++x) {
        const int32_t qr = (int32_t)(qrow_base + (int64_t)(qa + x) * kPfTile);
        tma_load_2d(base + kQOff + x * kTileBytes, &tq, 0, qr, q_full);
        tma_load_2d(base + kQOff + x * kTileBytes + 16384, &tq, 64, qr, q_full);
      }
      // K tiles are freed by their S products, V tiles by their P V products: two rings, filled in
      // tile order (K_j, V_j, K_j+1, ...)
      int kfills = 0, vfills = 0;
      for (int j = 0; j < nt; ++j) {
        const int s = j & 1;
        const int32_t kr = (int32_t)(krow0 + (int64_t)j * kPfTile);
        if (pf_aborted(flag) || !mbar_wait(k_empty(s), ((j >> 1) & 1) ^ 1)) { pf_fail(a, flag, kPfProducer); break; }
        mbar_expect_tx(k_full(s), 32768);
        tma_load_2d(base + kKOff + s * kTileBytes, &tk, 0, kr, k_full(s));
        tma_load_2d(base + kKOff + s * kTileBytes + 16384, &tk, 64, kr, k_full(s));
        ++kfills;
        if (pf_aborted(flag) || !mbar_wait(v_empty(s), ((j >> 1) & 1) ^ 1)) { pf_fail(a, flag, kPfProducer); break; }
        mbar_expect_tx(v_full(s), 32768);
        tma_load_2d(base + kVOff + s * kTileBytes, &tv, 0, kr, v_full(s));
        tma_load_2d(base + kVOff + s * kTileBytes + 16384, &tv, 64, kr, v_full(s));
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
    // The K (V) tile of the last step is read by tile B alone: its stage sees one of nq releases,
    // and is never refilled.
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(128, 128);
      constexpr uint32_t idesc_o = umma_idesc_bf16(128, 128) | kUmmaBMajorMN;
      const int ntA = nt_x[0], ntB = nq == 2 ? nt_x[1] : 0;
      bool ok = pf_wait(q_full, 0, flag);
      bool issued = false;
      // S_x(j) may start once K_j has landed and the tile's P V product of step j - 1 (which reads
      // the same TMEM columns) has completed; P_x(j) V_j once V_j has landed and the softmax has
      // written P_x(j).  The tile load is waited for first (it has normally landed long before), and
      // not again by the second tile that reads it.
      auto s_ready = [&](int x, int j) {
        const bool k_seen = x == 1 && j < ntA;
        return (k_seen || pf_wait(k_full(j & 1), (j >> 1) & 1, flag)) &&
               (j == 0 || pf_wait(pv_done(x), (j - 1) & 1, flag));
      };
      auto pv_ready = [&](int x, int j) {
        const bool v_seen = x == 1 && j < ntA;
        return (v_seen || pf_wait(v_full(j & 1), (j >> 1) & 1, flag)) && pf_wait(p_full(x), j & 1, flag);
      };
      auto s_step = [&](int x, int j, int kk) {
        const uint32_t sq = base + kQOff + x * kTileBytes, sk = base + kKOff + (j & 1) * kTileBytes;
        const uint32_t kb = kk >> 2, off = (kk & 3) * 32;
        umma_bf16(tmem + x * kTileCols + kSCol, umma_desc_sw128(sq + kb * 16384 + off),
                  umma_desc_sw128(sk + kb * 16384 + off), idesc_s, kk > 0);
      };
      auto pv_step = [&](int x, int j, int kk) {
        const uint32_t sv = base + kVOff + (j & 1) * kTileBytes;
        umma_bf16_ta(tmem + x * kTileCols + kOCol, tmem + x * kTileCols + kSCol + kk * 8,
                     umma_desc_sw128_mn(sv + kk * 2048, 16384), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
      };
      // a commit tracks every product issued before it, so each signals no earlier than its own
      auto s_issued = [&](int x, int j) {
        umma_commit(s_full(x));
        umma_commit(k_empty(j & 1));
        issued = true;
      };
      auto pv_issued = [&](int x, int j) {
        umma_commit(pv_done(x));
        umma_commit(v_empty(j & 1));
      };
      auto s_alone = [&](int x, int j) -> bool {
        if (!s_ready(x, j)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) s_step(x, j, kk);
        s_issued(x, j);
        return true;
      };
      ok = ok && s_alone(0, 0);
      if (ntB > 0) ok = ok && s_alone(1, 0);
      for (int j = 0; j < nt && ok; ++j) {
        if (j < ntA) {
          if (!(ok = pv_ready(0, j))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kPfTile / 16; ++kk) pv_step(0, j, kk);
          pv_issued(0, j);
        }
        const bool pvb = j < ntB, sa = j + 1 < ntA;
        if (pvb && !(ok = pv_ready(1, j))) break;
        if (sa && !(ok = s_ready(0, j + 1))) break;
        if (pvb || sa) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            if (pvb) pv_step(1, j, kk);
            if (sa) s_step(0, j + 1, kk);
          }
          if (pvb) pv_issued(1, j);
          if (sa) s_issued(0, j + 1);
        }
        if (j + 1 < ntB) ok = s_alone(1, j + 1);
      }
      if (!ok) pf_fail(a, flag, kPfMma);
      if (issued) {
        umma_commit(drain);
        if (!mbar_wait(drain, 0)) set_device_error(a.err, KVSEL_ERR_TIMEOUT, kPfDrain);
      }
    }
  } else {
    // softmax / epilogue: warpgroup x = tile, thread = query row of the tile
    const int x = (warp - 2) / 4;
    const int quarter = warp % 4;
    const int row = quarter * 32 + lane;
    const int qt = qa + x;
    const int i = qt * kPfTile + row;                               // row index in the sequence
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16) + x * kTileCols;
    const float scale = a.scale_log2;
    const int ntx = x < nq ? nt_x[x] : 0;
    float m = -INFINITY, l = 0.f;
    bool ok = x < nq;
    for (int j = 0; j < ntx; ++j) {
      ok = __all_sync(0xffffffffu, ok && pf_wait(s_full(x), j & 1, flag));
      if (!ok) {
        if (lane == 0) pf_fail(a, flag, kPfSoftmax);
        break;
      }
      tc_fence_after();
      const bool diag = j == ntx - 1;
      // both halves of the S row; P then goes over the columns already read (keys 0..63 into
      // columns 0..31, keys 64..127 into 32..63), packed in place into the same registers
      uint32_t rv[64], rw[64];
      tmem_ld64_async(lane_base + kSCol + 64, rv);
      tmem_ld64_async(lane_base + kSCol, rw);
      tmem_wait_ld64(rv);                                      // one wait covers both loads
      reg_tie64(rw);
      float* v = reinterpret_cast<float*>(rv);
      float* w = reinterpret_cast<float*>(rw);
      if (diag) {
        mask64(v, j * kPfTile + 64, i);
        mask64(w, j * kPfTile, i);
      }
      const float mt = fmaxf(max64(v), max64(w)) * scale;         // scale > 0: max commutes
      // lazy rescale: the exponent offset moves only when the tile's max exceeds it by more than 2^8
      float alpha = 1.f;
      if (mt > m + 8.f) {
        alpha = m == -INFINITY ? 0.f : fast_ex2(m - mt);
        m = mt;
      }
      const float2 sc = make_float2(scale, scale), nm = make_float2(-m, -m);
      float sum = exp_pack64(w, sc, nm, rw);
      tmem_st32(lane_base + kSCol, rw);
      sum += exp_pack64(v, sc, nm, rv);
      tmem_st32(lane_base + kSCol + 32, rv);
      l = l * alpha + sum;
      // O is final for tile j - 1 here (this tile's S was issued after that P V product completed)
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        uint32_t* r = rv;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          tmem_ld64_async(lane_base + kOCol + hh * 64, r);
          tmem_wait_ld64(r);
#pragma unroll
          for (int c = 0; c < 64; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
          tmem_st64(lane_base + kOCol + hh * 64, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(x));
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, !pf_aborted(flag) && mbar_wait(pv_done(x), (ntx - 1) & 1));
      if (!ok && lane == 0) pf_fail(a, flag, kPfSoftmax);
    }
    if (ok) {
      tc_fence_after();
      uint32_t r[64];
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool live = i < N;
      const int64_t qrow = qrow_base + i;
      __nv_bfloat16* orow = a.o + qrow * D;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        tmem_ld64_async(lane_base + kOCol + hh * 64, r);
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
            *reinterpret_cast<uint4*>(orow + hh * 64 + c * 8) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (live) {
        const float lse2 = m + log2f(l);
        if (a.lse != nullptr) a.lse[qrow] = lse2 * 0.6931471805599453f;
        if (i >= si.L) {                                            // an observation-window row
          const int jw = i - si.L, hl = h - g * a.G;
          const int64_t unit = ((int64_t)b * a.n_layers + layer) * a.h_kv + g;
          a.lse_win[unit * (a.G * a.W) + hl * a.W + jw] = lse2;
          const uint4* src = reinterpret_cast<const uint4*>(a.q + qrow * D);
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
    const int64_t n = t.s[b].n_keys;
    q_rows += (int64_t)d.n_layers * d.h_q * n;
    k_rows += (int64_t)d.n_layers * d.h_kv * n;
    nmax = n > nmax ? n : nmax;
  }
  if (q_rows + kPfTile >= (int64_t(1) << 31) || k_rows + kPfTile >= (int64_t(1) << 31)) return KVSEL_ERR_UNSUPPORTED;
  a.n_pairs = (int32_t)((nmax + 2 * kPfTile - 1) / (2 * kPfTile));
  CUtensorMap tq, tk, tv;
  if (!pf_map(&tq, q, q_rows) || !pf_map(&tk, k, k_rows) || !pf_map(&tv, v, k_rows)) return KVSEL_ERR_CUDA;
  if (set_smem((const void*)prefill_kernel, kPfSmem) != cudaSuccess) return KVSEL_ERR_CUDA;
  const int64_t grid = (int64_t)a.n_pairs * d.batch * d.n_layers * d.h_q;
  if (grid >= (int64_t(1) << 31)) return KVSEL_ERR_UNSUPPORTED;
  TraceScope ts("prefill_tc", s);
  prefill_kernel<<<(unsigned)grid, kPfThreads, kPfSmem, s>>>(tq, tk, tv, a, t);
  return launch_status();
}

}  // namespace kvsel
