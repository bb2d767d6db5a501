// Window-attention scoring on the 5th-generation tensor cores (tcgen05 / TMEM), sm_103a.
//
// Same two passes as the CUDA-core version (ClusterAttn, 'Background and key
// observations': masked window softmax over the full row, column sum over the
// window rows for prefix columns), with the logits of each 128-key tile made
// by UMMA from TMA-staged operands:
//
//   pass 1  rows on TMEM lanes:  D[128 rows x 128 keys] = Q · K_tileᵀ; each
//           epilogue thread owns one window row and keeps an online max / sum.
//   pass 2  keys on TMEM lanes:  D[128 keys x RT rows] = K_tile · Qᵀ; each
//           epilogue thread owns one key and sums 2^(z·log2e/√d − lse) over the
//           rows of each head in registers (no cross-lane reduction), then the
//           group reduce, max-pool and page reduce run on the segment in smem.
//
// Persistent CTAs (one per SM).  Pass 1 walks a contiguous range of (unit,
// segment) work items; pass 2 takes an equal share of all units' prefix pages
// laid end to end, cut into pieces at unit ends and every kSeg2Max keys, so
// that every CTA emits the same number of pages however many units there are.  Warp roles: warp 0 issues TMA (Q once per unit, K
// tiles through an NK-stage ring), warp 1 owns TMEM and issues UMMA into a
// ring of TMEM accumulators, warps 2.. are the epilogue (8 warps; 16 in pass 1
// over 256 rows).  All hand-offs are
// mbarriers with bounded waits; a wait that gives up records
// KVSEL_ERR_TIMEOUT in the workspace error word and the CTA unwinds.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "sm100.cuh"

namespace kvsel {
namespace {

using namespace sm100;

constexpr int kTileKeys = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kEpiBarrier = 1;   // named barrier id of the epilogue warps

enum : uint32_t { kWhereProducer = 1, kWhereMma = 2, kWhereEpilogue = 3, kWhereDrain = 4 };

// Prefix keys per pass-2 segment (rounded down to whole pages): the segment's scores are held in
// shared memory until it is pooled.
constexpr int kSeg2Max = 8192;

// Shared-memory plan (offsets from a 1024-byte aligned base).
template <bool PASS2, int RT, int D, int NK>
struct Plan {
  static constexpr int kDBlocks = D / 64;                   // 128-byte swizzle atoms along d
  static constexpr uint32_t kQBlock = RT * 128;             // one d-block of Q: RT rows x 128 B
  static constexpr uint32_t kQBytes = kQBlock * kDBlocks;
  static constexpr uint32_t kKBlock = kTileKeys * 128;      // one d-block of a K tile
  static constexpr uint32_t kKBytes = kKBlock * kDBlocks;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKOff = kQOff + kQBytes;
  // With 256 rows, pass 2 adds each row's -lse to its logits on the tensor cores: one more K = 16
  // product of a block of ones (128 keys) with the rows' -lse / scale split into bf16 parts.
  static constexpr bool kFold = PASS2 && RT == 256;
  // Epilogue warps: 8, or 16 over 256 rows (four warps per TMEM lane quarter, so that every SM
  // sub-partition has four warps' exponentials in flight).  Over 256 rows the two pairs of
  // warpgroups take alternate tiles (one TMEM stage each), so only one pair's warps release a stage.
  static constexpr int kEW = RT == 256 ? 16 : 8;
  static constexpr int kThreads = 32 * (2 + kEW);
  static constexpr int kStageReaders = RT == 256 ? kEW / 2 : kEW;
  static constexpr uint32_t kOnesOff = kKOff + NK * kKBytes;                // 128 rows x 32 B of bf16 ones
  static constexpr uint32_t kCOff = kOnesOff + (kFold ? 128 * 32 : 0);     // RT rows x 32 B
  static constexpr uint32_t kSsOff = kCOff + (kFold ? RT * 32 : 0);        // pass-2 segment scores
  static constexpr uint32_t kSsFloats = PASS2 ? kSeg2Max + 128 : 0;
  static constexpr uint32_t kLseOff = kSsOff + kSsFloats * 4;             // pass-2 row lse (RT floats)
  static constexpr uint32_t kRedOff = kLseOff + (PASS2 ? RT * 4 : 0);     // pass-1 (m, l) exchange
  static constexpr uint32_t kNT = kTmemCols / RT;                         // TMEM accumulator stages
  static constexpr uint32_t kBarOff = kRedOff + (PASS2 ? 0 : 128 * 8);   // 128 rows' (m, l) per exchange round
  // barriers: full[NK], empty[NK], tfull[NT], tempty[NT], q_full, q_empty, drain
  static constexpr uint32_t kNumBars = 2 * NK + 2 * kNT + 3;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;            // tmem slot, abort flag
  static constexpr uint32_t kBytes = kMiscOff + 16;
  static constexpr size_t kSmem = kBytes + 1024;                          // + alignment slack
  static_assert(kSmem <= 227 * 1024, "shared memory plan too large");
};

struct TcArgs {
  ScoreShape sh;
  float* scores;
  float* page_scores;
  float* lse;
  float2* part;
  DeviceError* err;
};

// Geometry of one work item.
struct Item {
  int b, ul, seg, layer, g;
  int unit;            // global (sequence, layer, KV head) unit index
  int L, n_keys;
  int32_t q_row0;      // first Q row of the unit's group in the 2-D Q view
  int32_t k_row0;      // first K row of the unit in the 2-D K view
  int ta, tb;          // key range whose tiles are processed
  int a0, a1;          // pass 2: prefix range whose scores are emitted
};

// Tile row r of a unit: with heads padded to Wp rows, row r is window row j = r % Wp of head
// h = r / Wp, a real row when j < W and h < G, whose index among the unit's R = G W rows is h W + j;
// without padding (Wp == W) tile row r is row r.  -1 for a padding row.
__device__ __forceinline__ int real_row(const ScoreShape& sh, int r) {
  if (sh.Wp == sh.W) return r < sh.R ? r : -1;
  const int h = r / sh.Wp, j = r - h * sh.Wp;
  return (j < sh.W && h < sh.G) ? h * sh.W + j : -1;
}

// Heads of the group that start at tile row c0 or later (the head sums of a 64-column block that
// begins there), for the group max: the blocks' remaining heads are all padding rows.
__device__ __forceinline__ int heads_from(const ScoreShape& sh, int c0) {
  const int hw = sh.Wp < 64 ? sh.Wp : 64;
  return max(0, sh.G - c0 / hw);
}

// Unit ul of sequence b: the fields every item of it shares.
__device__ __forceinline__ void unit_fields(const SeqTable& t, const ScoreShape& sh, int b, int ul, Item& it) {
  const SeqInfo si = t.s[b];   // a copy: loads once, whatever the table lives in
  it.b = b;
  it.ul = ul;
  it.layer = ul / sh.h_kv;
  it.g = ul % sh.h_kv;
  it.unit = si.unit0 + ul;
  it.L = si.L;
  it.n_keys = si.n_keys;
  it.q_row0 = (int32_t)((((int64_t)b * sh.n_layers + it.layer) * sh.h_q + (int64_t)it.g * sh.G) * sh.W);
  it.k_row0 = (int32_t)(si.k_off / sh.d + ((int64_t)it.layer * sh.h_kv + it.g) * si.n_keys);
}

// This CTA's work, in order.  Pass 1: items [n*c/grid, n*(c+1)/grid) of the launch's (unit,
// segment) items.  Pass 2: the launch's units' prefix pages laid end to end (sequence b's units
// start at page item0, n_seg pages each), pages [n*c/grid, n*(c+1)/grid) of them, cut into
// pieces that end at a unit's end, at the share's end or after seg2 keys.
template <bool PASS2>
struct Work {
  int pos, end;
  __device__ __forceinline__ explicit Work(const SeqTable& t)
      : pos((int)(((int64_t)blockIdx.x * t.n_items) / gridDim.x)),
        end((int)(((int64_t)(blockIdx.x + 1) * t.n_items) / gridDim.x)) {}
  __device__ __forceinline__ bool next(const SeqTable& t, const ScoreShape& sh, Item& it) {
    if (pos >= end) return false;
    const int b = find_seq(t, pos);
    const SeqInfo si = t.s[b];   // a copy: loads once, whatever the table lives in
    const int local = pos - si.item0;
    if (!PASS2) {
      unit_fields(t, sh, b, local / si.n_seg, it);
      it.seg = local % si.n_seg;
      it.ta = it.seg * sh.seg1;
      it.tb = min(si.n_keys, it.ta + sh.seg1);
      it.a0 = it.a1 = 0;
      pos += 1;
    } else {
      unit_fields(t, sh, b, local / si.n_seg, it);
      const int pin = local % si.n_seg;                       // first page of the piece in its unit
      const int n = min(min(si.n_seg - pin, sh.seg2 / sh.page_size), end - pos);
      const int pr = (sh.pool_k - 1) / 2;
      it.seg = pin;
      it.a0 = pin * sh.page_size;
      it.a1 = min(si.L, (pin + n) * sh.page_size);
      it.ta = max(0, it.a0 - pr);
      it.tb = min(si.L, it.a1 + pr);
      pos += n;
    }
    return true;
  }
  __device__ __forceinline__ int index() const { return pos - 1; }   // pass 1: the item just taken
};

__device__ __forceinline__ bool aborted(const volatile uint32_t* flag) { return *flag != 0; }

__device__ __forceinline__ void fail(const TcArgs& a, volatile uint32_t* flag, uint32_t where) {
  set_device_error(a.err, KVSEL_ERR_TIMEOUT, where);
  *flag = 1;
}

// ---------------------------------------------------------------- producer (warp 0)
// The rows' -lse / scale for the extra K = 16 product of pass 2 (256 rows): c / 2 as the sum of
// three bf16 parts p1 + p2 + p3 (24 significant bits), stored as [p1 p2 p3 0 0 0 0 0] in both
// 16-byte halves of the row's 32 bytes, so that the product with a row of ones gives c whichever
// way the 32-byte swizzle permutes the halves.  Padding rows get c = -2^101: their p is 0.
// Each lane writes rows lane, lane + 32, ...; the writes are made visible to the tensor cores'
// operand reads before the warp's leader signals the unit's Q tile.
template <int RT>
__device__ __forceinline__ void write_fold_rows(const TcArgs& a, int unit, uint8_t* crow, int lane) {
  const double inv = 1.0 / (double)a.sh.scale_log2;
  for (int r = lane; r < RT; r += 32) {
    __nv_bfloat16 p1, p2, p3;
    const int rr = real_row(a.sh, r);
    if (rr >= 0) {
      const double h = -0.5 * (double)a.lse[(int64_t)unit * a.sh.R + rr] * inv;
      p1 = __float2bfloat16_rn((float)h);
      const double r1 = h - (double)__bfloat162float(p1);
      p2 = __float2bfloat16_rn((float)r1);
      p3 = __float2bfloat16_rn((float)(r1 - (double)__bfloat162float(p2)));
    } else {
      p1 = __float2bfloat16_rn(-0x1p100f);
      p2 = p3 = __float2bfloat16_rn(0.f);
    }
    const uint32_t w0 = (uint32_t)__bfloat16_as_ushort(p1) | ((uint32_t)__bfloat16_as_ushort(p2) << 16);
    const uint32_t w1 = (uint32_t)__bfloat16_as_ushort(p3);
    uint4* dst = reinterpret_cast<uint4*>(crow + r * 32);
    dst[0] = make_uint4(w0, w1, 0u, 0u);
    dst[1] = make_uint4(w0, w1, 0u, 0u);
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// Lane 0 issues every TMA load and does every wait; the whole warp runs the loop (its decisions
// are lane 0's, broadcast) so that all lanes can write the pass-2 row constants at a unit change.
template <bool PASS2, int RT, int D, int NK>
__device__ void produce(const CUtensorMap* tq, const CUtensorMap* tqh, const CUtensorMap* tk, const TcArgs& a,
                        const SeqTable& t, uint32_t base, uint8_t* sbase, volatile uint32_t* flag) {
  using P = Plan<PASS2, RT, D, NK>;
  const int lane = threadIdx.x % 32;
  const bool leader = lane == 0;
  const bool fold = P::kFold && PASS2 && !a.sh.logits;
  const uint32_t bars = base + P::kBarOff;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (NK + s); };
  const uint32_t q_full = bars + 8u * (2 * NK + 2 * P::kNT);
  const uint32_t q_empty = q_full + 8;
  if (leader) {
    tma_prefetch_desc(tq);
    tma_prefetch_desc(tk);
  }
  int ks = 0;
  uint32_t kph = 0, qph = 0;
  uint32_t n_fills = 0, n_q = 0;
  int prev_unit = -1;
  Work<PASS2> work(t);
  Item it;
  while (__shfl_sync(0xffffffffu, leader && !aborted(flag) ? 1 : 0, 0) && work.next(t, a.sh, it)) {
    if (it.unit != prev_unit) {
      int ok = 1;
      if (leader) ok = mbar_wait(q_empty, qph ^ 1) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        if (leader) fail(a, flag, kWhereProducer);
        break;
      }
      if (fold) write_fold_rows<RT>(a, it.unit, sbase + P::kCOff, lane);
      if (leader) {
        if (a.sh.Wp == a.sh.W) {
          mbar_expect_tx(q_full, P::kQBytes);
#pragma unroll
          for (int db = 0; db < P::kDBlocks; ++db)
#pragma unroll
            for (int m = 0; m < RT / 128; ++m)
              tma_load_2d(base + P::kQOff + db * P::kQBlock + m * 16384, tq, db * 64, it.q_row0 + m * 128, q_full);
        } else {
          // padded heads: head h's rows land at tile rows h Wp .. (boxes of Wp rows; the rows past a
          // head's W are the next head's, and count as padding)
          mbar_expect_tx(q_full, (uint32_t)(a.sh.G * a.sh.Wp * 128 * P::kDBlocks));
          for (int db = 0; db < P::kDBlocks; ++db)
            for (int h = 0; h < a.sh.G; ++h) {
              const int r0 = h * a.sh.Wp;
              tma_load_2d(base + P::kQOff + db * P::kQBlock + (r0 >> 7) * 16384 + (r0 & 127) * 128, tqh, db * 64,
                          it.q_row0 + h * a.sh.W, q_full);
            }
        }
      }
      qph ^= 1;
      ++n_q;
      prev_unit = it.unit;
    }
    int ok = 1;
    if (leader) {
      for (int t0 = it.ta; t0 < it.tb; t0 += kTileKeys) {
        if (!mbar_wait(empty(ks), kph ^ 1)) { ok = 0; break; }
        mbar_expect_tx(full(ks), P::kKBytes);
        const uint32_t dst = base + P::kKOff + ks * P::kKBytes;
#pragma unroll
        for (int db = 0; db < P::kDBlocks; ++db)
          tma_load_2d(dst + db * P::kKBlock, tk, db * 64, it.k_row0 + t0, full(ks));
        ++n_fills;
        if (++ks == NK) { ks = 0; kph ^= 1; }
      }
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) {
      if (leader) fail(a, flag, kWhereProducer);
      break;
    }
  }
  if (!leader) return;
  // Loads still in flight (possible only after an abort) must land before the CTA exits:
  // wait for the phase of each stage's last fill (returns at once when already complete).
  for (int s = 0; s < NK; ++s) {
    if (n_fills > (uint32_t)s) {
      const uint32_t cnt = (n_fills - s + NK - 1) / NK;
      if (!mbar_wait(full(s), (cnt - 1) & 1)) set_device_error(a.err, KVSEL_ERR_TIMEOUT, kWhereDrain);
    }
  }
  if (n_q > 0 && !mbar_wait(q_full, (n_q - 1) & 1)) set_device_error(a.err, KVSEL_ERR_TIMEOUT, kWhereDrain);
}

// ---------------------------------------------------------------- MMA issuer (one thread)
template <bool PASS2, int RT, int D, int NK>
__device__ void issue_mma(const TcArgs& a, const SeqTable& t, uint32_t base, uint32_t tmem,
                          volatile uint32_t* flag) {
  using P = Plan<PASS2, RT, D, NK>;
  const uint32_t bars = base + P::kBarOff;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (NK + s); };
  auto tfull = [&](int s) { return bars + 8u * (2 * NK + s); };
  auto tempty = [&](int s) { return bars + 8u * (2 * NK + P::kNT + s); };
  const uint32_t q_full = bars + 8u * (2 * NK + 2 * P::kNT);
  const uint32_t q_empty = q_full + 8;
  const uint32_t drain = q_empty + 8;
  // pass 1: M = 128 window rows (per M block), N = 128 keys;  pass 2: M = 128 keys, N = RT rows
  constexpr uint32_t idesc = PASS2 ? umma_idesc_bf16(128, RT) : umma_idesc_bf16(128, 128);
  const bool fold = P::kFold && PASS2 && !a.sh.logits;
  int ks = 0, ts = 0;
  uint32_t kph = 0, tph = 0, qph = 0;
  int prev_unit = -1;
  bool issued = false;
  Work<PASS2> work(t);
  for (Item it; !aborted(flag) && work.next(t, a.sh, it);) {
    if (it.unit != prev_unit) {
      if (prev_unit >= 0) umma_commit(q_empty);     // previous unit's Q is free once its MMAs finish
      if (!mbar_wait(q_full, qph)) { fail(a, flag, kWhereMma); break; }
      qph ^= 1;
      prev_unit = it.unit;
    }
    bool ok = true;
    for (int t0 = it.ta; t0 < it.tb; t0 += kTileKeys) {
      if (!mbar_wait(full(ks), kph) || !mbar_wait(tempty(ts), tph ^ 1)) { ok = false; break; }
      tc_fence_after();
      const uint32_t kbase = base + P::kKOff + ks * P::kKBytes;
      const uint32_t qbase = base + P::kQOff;
      const uint32_t d_tmem = tmem + ts * RT;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t db = kk >> 2, off = (kk & 3) * 32;
        if (PASS2) {
          umma_bf16(d_tmem, umma_desc_sw128(kbase + db * P::kKBlock + off),
                    umma_desc_sw128(qbase + db * P::kQBlock + off), idesc, kk > 0);
        } else {
#pragma unroll
          for (int m = 0; m < RT / 128; ++m)
            umma_bf16(d_tmem + m * 128, umma_desc_sw128(qbase + db * P::kQBlock + m * 16384 + off),
                      umma_desc_sw128(kbase + db * P::kKBlock + off), idesc, kk > 0);
        }
      }
      if (fold)   // + (-lse / scale) of every row: ones (keys) x the rows' constants
        umma_bf16(d_tmem, umma_desc_sw32(base + P::kOnesOff), umma_desc_sw32(base + P::kCOff), idesc, 1);
      issued = true;
      umma_commit(empty(ks));     // K stage free once these MMAs have read it
      umma_commit(tfull(ts));     // accumulator ready for the epilogue
      if (++ks == NK) { ks = 0; kph ^= 1; }
      if (++ts == (int)P::kNT) { ts = 0; tph ^= 1; }
    }
    if (!ok) { fail(a, flag, kWhereMma); break; }
  }
  // Every MMA issued must be complete before TMEM is released.
  if (issued) {
    umma_commit(drain);
    if (!mbar_wait(drain, 0)) set_device_error(a.err, KVSEL_ERR_TIMEOUT, kWhereDrain);
  }
}

// ---------------------------------------------------------------- epilogue helpers
template <int EW>
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync %0, %1;" ::"r"(kEpiBarrier), "r"(32 * EW) : "memory");
}

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Epilogue arithmetic on 64 accumulator columns, written for instruction-level parallelism and
// issue economy: packed fp32x2 FMA / add (two columns per instruction), three-input max, and
// independent partial results combined by a fixed pairwise tree (so results do not depend on
// scheduling); invisible columns enter as -inf.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float2 ex2x2(float2 x) { return make_float2(fast_ex2(x.x), fast_ex2(x.y)); }

template <int N>
__device__ __forceinline__ float tree_sum(float* a) {
#pragma unroll
  for (int w = N / 2; w >= 1; w /= 2)
#pragma unroll
    for (int i = 0; i < w; ++i) a[i] += a[i + w];
  return a[0];
}

template <int N>
__device__ __forceinline__ float tree_sum2(float2* a) {
#pragma unroll
  for (int w = N / 2; w >= 1; w /= 2)
#pragma unroll
    for (int i = 0; i < w; ++i) a[i] = __fadd2_rn(a[i], a[i + w]);
  return a[0].x + a[0].y;
}

__device__ __forceinline__ float max64(const float* v) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float* c = v + 8 * k;
    m[k] = fmaxf(fmax3(fmax3(c[0], c[1], c[2]), c[3], c[4]), fmax3(c[5], c[6], c[7]));
  }
  return fmax3(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// sum_i 2^(v_i * scale + off)
__device__ __forceinline__ float expsum64(const float* v, float scale, float off) {
  const float2 sc = make_float2(scale, scale), of = make_float2(off, off);
  float2 a[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) a[k] = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 32; ++i)
    a[i & 3] = __fadd2_rn(a[i & 3], ex2x2(__ffma2_rn(make_float2(v[2 * i], v[2 * i + 1]), sc, of)));
  return tree_sum2<4>(a);
}

// Exponent argument of a column pair: v * scale + nl (FOLDED: the -lse is already in v).
template <bool FOLDED>
__device__ __forceinline__ float2 exp_arg2(float v0, float v1, float2 sc, const float2* nl, int i) {
  if constexpr (FOLDED) return __fmul2_rn(make_float2(v0, v1), sc);
  else return __ffma2_rn(make_float2(v0, v1), sc, nl[i]);
}

// Column mass of 64 rows for one key: sum (MAXW = 0) or max over heads of MAXW rows of
// sum_i 2^(v_i * scale + nl_i), nl = -lse of each row as pairs (FOLDED: v_i * scale alone,
// the accumulator already holding z - lse / scale).
template <int MAXW, bool FOLDED = false>
__device__ __forceinline__ float colmass64(const float* v, const float2* nl, float scale) {
  const float2 sc = make_float2(scale, scale);
  if constexpr (MAXW == 0) {
    float2 a[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) a[k] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      a[i & 3] = __fadd2_rn(a[i & 3], ex2x2(exp_arg2<FOLDED>(v[2 * i], v[2 * i + 1], sc, nl, i)));
    return tree_sum2<4>(a);
  } else {
    constexpr int HW = MAXW < 64 ? MAXW : 64;      // rows per head
    constexpr int NP = HW / 2;                     // pairs per head
    constexpr int NA = NP < 4 ? NP : 4;
    float red = 0.f;
#pragma unroll
    for (int h = 0; h < 64 / HW; ++h) {
      float2 a[NA];
#pragma unroll
      for (int k = 0; k < NA; ++k) a[k] = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const int c = h * NP + i;
        a[i % NA] = __fadd2_rn(a[i % NA], ex2x2(exp_arg2<FOLDED>(v[2 * c], v[2 * c + 1], sc, nl, c)));
      }
      red = fmaxf(red, tree_sum2<NA>(a));
    }
    return red;
  }
}

// Logits mode: the same reductions over sum_i v_i * w_i, w = 1/sqrt(d) for real rows and 0 for
// the padding rows (GemFilter's pre-softmax score; no exponentials).
template <int MAXW>
__device__ __forceinline__ float linmass64(const float* v, const float2* w, int nh = 64) {
  if constexpr (MAXW == 0) {
    float2 a[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) a[k] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 32; ++i) a[i & 3] = __ffma2_rn(make_float2(v[2 * i], v[2 * i + 1]), w[i], a[i & 3]);
    return tree_sum2<4>(a);
  } else {
    constexpr int HW = MAXW < 64 ? MAXW : 64;
    constexpr int NP = HW / 2;
    constexpr int NA = NP < 4 ? NP : 4;
    float red = -INFINITY;
#pragma unroll
    for (int h = 0; h < 64 / HW; ++h) {
      float2 a[NA];
#pragma unroll
      for (int k = 0; k < NA; ++k) a[k] = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const int c = h * NP + i;
        a[i % NA] = __ffma2_rn(make_float2(v[2 * c], v[2 * c + 1]), w[c], a[i % NA]);
      }
      // heads past the group's last (all padding) have no sum: a zero would outrank negative maxima
      if (h < nh) red = fmaxf(red, tree_sum2<NA>(a));
    }
    return red;
  }
}

// Online (offset, sum) update of one row with 64 new columns, the first nvis of them visible:
// l = sum of 2^(z scale - m).  Once the row has an offset m, the exponentials are taken against
// it without forming the new columns' maximum: when their sum s is at most 2^8 every term is, so
// no column lies more than 8 above the offset and s is added as it is.  A larger (or infinite) s
// moves the offset to the columns' maximum, which is then at least m + 2 (64 terms of at most
// 2^(max - m) exceed 2^8), and the sum is rescaled and retaken.  The row's log-sum-exp
// m + log2 l is the same whichever offset the sum was taken against.
__device__ __forceinline__ void online_update64(float* v, int nvis, float scale, float& m, float& l) {
  if (nvis < 64) {
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if (i >= nvis) v[i] = -INFINITY;
  }
  if (m == -INFINITY) {                     // first visible columns of the row in this segment
    const float mx = max64(v);
    if (mx > -INFINITY) {
      m = mx * scale;
      l = expsum64(v, scale, -m);
    }
    return;
  }
  const float s = expsum64(v, scale, -m);
  if (s <= 256.f) {
    l += s;
  } else {
    const float mx = max64(v) * scale;
    l = l * fast_ex2(m - mx) + expsum64(v, scale, -mx);
    m = mx;
  }
}

// Epilogue thread geometry: warps 2..; warp w may read TMEM lanes 32*(w%4) .. +31.
struct EpiThread {
  int wg;        // epilogue warpgroup 0 .. (epilogue warps / 4) - 1
  int quarter;   // TMEM lane quarter
  int lane;
  int lrow;      // TMEM lane = quarter * 32 + lane
  int etid;      // 0 .. (epilogue threads) - 1
};

__device__ __forceinline__ EpiThread epi_thread() {
  EpiThread e;
  const int warp = threadIdx.x / 32;
  e.wg = (warp - 2) / 4;
  e.quarter = warp % 4;
  e.lane = threadIdx.x % 32;
  e.lrow = e.quarter * 32 + e.lane;
  e.etid = threadIdx.x - 64;
  return e;
}

// Whether the accumulator stage (bar, parity) may be read.  `ready` is the previous tile's
// non-blocking probe of it, issued before that tile's arithmetic so that its latency overlaps the
// arithmetic; otherwise the warp waits (bounded), reading the abort flag only then.  The tensor-
// memory loads that follow are warp-collective, so the decision is the warp's.
__device__ __forceinline__ bool tile_ready(bool ready, uint32_t bar, uint32_t parity, volatile uint32_t* flag) {
  if (__all_sync(0xffffffffu, ready)) return true;
  return __all_sync(0xffffffffu, !aborted(flag) && mbar_wait(bar, parity));
}

// ---------------------------------------------------------------- pass 1 epilogue
// RT = 128: both warpgroups see all 128 rows, warpgroup e takes tile columns [64e, 64e + 64) of
// every tile (the next tile's accumulator probed before this tile's arithmetic).
// RT = 256: the pairs of warpgroups (0, 1) and (2, 3) take alternate tiles, pair p those this CTA
// takes at positions of parity p, always from TMEM stage p; warpgroup e takes rows
// 128 (e % 2) .. + 127 (accumulator block e % 2), all 128 columns as two 64-column halves.  The
// pairs run a tile apart, so one pair's waits and loads overlap the other's arithmetic.
// Either way each row has two partial (offset, sum)s, merged once per segment through shared
// memory (one exchange per 128 rows).
template <int RT, int D, int NK>
__device__ void epilogue_pass1(const TcArgs& a, const SeqTable& t, uint32_t base, uint8_t* sbase,
                               uint32_t tmem, volatile uint32_t* flag) {
  using P = Plan<false, RT, D, NK>;
  constexpr int EW = P::kEW;
  static_assert(EW / 4 * 64 * 128 == RT * kTileKeys, "every (row, column) of a tile has one thread");
  const EpiThread e = epi_thread();
  const uint32_t bars = base + P::kBarOff;
  auto tfull = [&](int s) { return bars + 8u * (2 * NK + s); };
  auto tempty = [&](int s) { return bars + 8u * (2 * NK + P::kNT + s); };
  constexpr bool kPairs = RT == 256;
  const int rblk = kPairs ? (e.wg & 1) : 0;                    // accumulator block (128 rows)
  const int chalf = e.wg >> (kPairs ? 1 : 0);                  // RT = 256: pair; else 64-column half
  const int trow = e.lrow + 128 * rblk;                         // tile row
  const int row = real_row(a.sh, trow);                         // the unit's row (-1: padding)
  const uint32_t col0 = kPairs ? 128u * rblk : 64u * chalf;    // TMEM column within a stage
  const int key0 = kPairs ? 0 : 64 * chalf;                    // tile key of that column
  float* red = reinterpret_cast<float*>(sbase + P::kRedOff);
  const float scale = a.sh.scale_log2;
  const bool rvalid = row >= 0;
  int ts = 0, nt = 0;                                           // nt: tiles this CTA has taken so far
  uint32_t tph = 0;
  Work<false> work(t);
  for (Item it; work.next(t, a.sh, it);) {
    const int item = work.index();
    const int row_last = it.L + (rvalid ? row % a.sh.W : 0);     // last key this row sees
    const int vis_end = min(it.tb, row_last + 1);
    float m = -INFINITY, l = 0.f;
    bool ready = false;      // this tile's accumulator was seen complete by the previous tile's probe
    for (int t0 = it.ta; t0 < it.tb; t0 += kTileKeys) {
      if constexpr (kPairs) {
        if ((nt++ & 1) != chalf) continue;
        // the tensor-memory loads below are warp-collective: decide per warp
        const bool ok = __all_sync(0xffffffffu, !aborted(flag) && mbar_wait(tfull(chalf), tph));
        tph ^= 1;
        if (!ok) {
          if (e.lane == 0) fail(a, flag, kWhereEpilogue);
          continue;
        }
        tc_fence_after();
        const uint32_t lane_base = tmem + ((uint32_t)(e.quarter * 32) << 16) + chalf * RT + col0;
        {
          float v[64];
          tmem_ld64(lane_base, v);
          if (rvalid) online_update64(v, vis_end - t0, scale, m, l);
        }
        {
          float v[64];
          tmem_ld64(lane_base + 64, v);
          tc_fence_before();
          __syncwarp();
          if (e.lane == 0) mbar_arrive(tempty(chalf));
          if (rvalid) online_update64(v, vis_end - (t0 + 64), scale, m, l);
        }
        continue;
      }
      const bool ok = tile_ready(ready, tfull(ts), tph, flag);
      if (!ok && e.lane == 0) fail(a, flag, kWhereEpilogue);
      float v[64];
      if (ok) {
        tc_fence_after();
        tmem_ld64(tmem + ((uint32_t)(e.quarter * 32) << 16) + ts * RT + col0, v);
        tc_fence_before();
        __syncwarp();
        if (e.lane == 0) mbar_arrive(tempty(ts));
      }
      if (++ts == (int)P::kNT) { ts = 0; tph ^= 1; }
      ready = t0 + kTileKeys < it.tb && mbar_test_wait(tfull(ts), tph);   // answer used at the next tile
      if (ok && rvalid) online_update64(v, vis_end - (t0 + key0), scale, m, l);
    }
    // per-row partial (m, l) of this segment: the second half's threads hand theirs over
#pragma unroll
    for (int rb = 0; rb < RT / 128; ++rb) {
      epi_sync<EW>();
      if (rblk == rb && chalf == 1) {
        red[2 * e.lrow] = m;
        red[2 * e.lrow + 1] = l;
      }
      epi_sync<EW>();
      if (rblk == rb && chalf == 0 && rvalid) {
        const float m2 = red[2 * e.lrow], l2 = red[2 * e.lrow + 1];
        const float M = fmaxf(m, m2);
        float S = 0.f;
        if (M > -INFINITY) S = (m > -INFINITY ? l * fast_ex2(m - M) : 0.f) + (m2 > -INFINITY ? l2 * fast_ex2(m2 - M) : 0.f);
        a.part[(int64_t)item * a.sh.R + row] = make_float2(M, S);
      }
    }
  }
}

// The group max of a key's two partials by shared-memory atomics: probabilities (>= 0) compare as
// their int bit patterns; the signed sums of pre-softmax scores compare through an order-preserving
// unsigned key (0 lies below every key), decoded in place before the segment is pooled.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ void max_into(float* slot, float v, bool signed_values) {
  if (signed_values) atomicMax(reinterpret_cast<unsigned int*>(slot), order_key(v));
  else atomicMax(reinterpret_cast<int*>(slot), __float_as_int(v));
}

// Pooling of a segment's group scores S[ta..tb) (the pooling halo included) into out[a0..a1), and,
// with P > 1, page reduce into pout over the pages of [a0, a1); every output is scaled by gscale
// (the 1 / (G W) of the mean reduce).  Window loads are independent of one another, so they
// overlap instead of forming a chain of shared-memory latencies.
__device__ __forceinline__ float window_max(const float* S, int ta, int tb, int tt, int pr) {
  float u = -INFINITY;
  if (pr <= 3) {
    float w[7];
#pragma unroll
    for (int x = 0; x < 7; ++x) {
      const int y = tt - 3 + x;
      w[x] = (x >= 3 - pr && x <= 3 + pr && y >= ta && y < tb) ? S[y - ta] : -INFINITY;
    }
    u = fmaxf(fmaxf(fmaxf(w[0], w[1]), fmaxf(w[2], w[3])), fmaxf(fmaxf(w[4], w[5]), w[6]));
  } else {
    const int lo = max(tt - pr, ta), hi = min(tt + pr, tb - 1);
#pragma unroll 8
    for (int y = lo; y <= hi; ++y) u = fmaxf(u, S[y - ta]);
  }
  return u;
}

// Mean over the in-range neighbours (the segment's halo reaches every in-range neighbour).
__device__ __forceinline__ float window_avg(const float* S, int ta, int tb, int tt, int pr) {
  const int lo = max(tt - pr, ta), hi = min(tt + pr, tb - 1);
  float acc = 0.f;
  if (pr <= 3) {
    float w[7];
#pragma unroll
    for (int x = 0; x < 7; ++x) {
      const int y = tt - 3 + x;
      w[x] = (y >= lo && y <= hi) ? S[y - ta] : 0.f;
    }
    acc = ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + w[6]);
  } else {
#pragma unroll 8
    for (int y = lo; y <= hi; ++y) acc += S[y - ta];
  }
  // a full window divides by the constant 2 pr + 1 (one multiply by its reciprocal); the segment's
  // first and last r positions by their own count
  const int cnt = hi - lo + 1;
  return cnt == 2 * pr + 1 ? acc * (1.0f / (float)(2 * pr + 1)) : acc / (float)cnt;
}

__device__ void pool_segment(const float* S, int ta, int tb, int a0, int a1, int pr, int P, int page_reduce,
                             int pool_type, float gscale, float* out, float* pout, int tid, int nthreads) {
  const bool avg = pool_type == KVSEL_POOL_AVG;
#pragma unroll 4
  for (int tt = a0 + tid; tt < a1; tt += nthreads)
    out[tt] = gscale * (avg ? window_avg(S, ta, tb, tt, pr) : window_max(S, ta, tb, tt, pr));
  if (P == 1) return;
  for (int p = a0 / P + tid; p * P < a1; p += nthreads) {
    const int lo = p * P, hi = min(a1, lo + P);
    float pv;
    if (page_reduce == KVSEL_REDUCE_MAX && !avg) {
      // the max over the page of the max-pooled scores is the max over the page widened by the window
      const int wlo = max(lo - pr, ta), whi = min(hi - 1 + pr, tb - 1);
      pv = -INFINITY;
#pragma unroll 8
      for (int y = wlo; y <= whi; ++y) pv = fmaxf(pv, S[y - ta]);
    } else if (page_reduce == KVSEL_REDUCE_MAX) {
      pv = -INFINITY;
      for (int tt = lo; tt < hi; ++tt) pv = fmaxf(pv, window_avg(S, ta, tb, tt, pr));
    } else {
      pv = 0.f;
      for (int tt = lo; tt < hi; ++tt) pv += avg ? window_avg(S, ta, tb, tt, pr) : window_max(S, ta, tb, tt, pr);
    }
    pout[p] = gscale * pv;
  }
}

// ---------------------------------------------------------------- pass 2 epilogue
// 128 rows, 8 epilogue warps: thread = key (TMEM lane); warpgroup e takes rows [64 e, 64 e + 64)
// (TMEM columns), whose -lse it holds in registers as column pairs.
// MAXW = 0: group sum (every row summed); otherwise group max with head width MAXW.
template <int RT, int D, int NK, int MAXW>
__device__ void epilogue_pass2(const TcArgs& a, const SeqTable& t, uint32_t base, uint8_t* sbase,
                               uint32_t tmem, volatile uint32_t* flag) {
  using P = Plan<true, RT, D, NK>;
  static_assert(RT == 128 && P::kEW == 8, "two warpgroups of 64 rows");
  constexpr int kEpiThreads = 32 * P::kEW;
  const EpiThread e = epi_thread();
  const uint32_t bars = base + P::kBarOff;
  auto tfull = [&](int s) { return bars + 8u * (2 * NK + s); };
  auto tempty = [&](int s) { return bars + 8u * (2 * NK + P::kNT + s); };
  float* Ss = reinterpret_cast<float*>(sbase + P::kSsOff);
  float* lse_s = reinterpret_cast<float*>(sbase + P::kLseOff);   // holds -lse per row
  const float scale = a.sh.scale_log2;
  const int col0 = e.wg * 64;
  const int pr = (a.sh.pool_k - 1) / 2;
  const int P_ = a.sh.page_size;
  int ts = 0;
  uint32_t tph = 0;
  Work<true> work(t);
  for (Item it; work.next(t, a.sh, it);) {
    epi_sync<P::kEW>();                                      // readers of the previous item are done
    for (int i = e.etid; i < it.tb - it.ta; i += kEpiThreads) Ss[i] = 0.f;
    for (int i = e.etid; i < RT; i += kEpiThreads) {
      const int rr = real_row(a.sh, i);
      if (a.sh.logits) lse_s[i] = rr >= 0 ? a.sh.scale_nat : 0.f;    // row weights of the logit sum
      else lse_s[i] = rr >= 0 ? -a.lse[(int64_t)it.unit * a.sh.R + rr] : -INFINITY;   // padding rows: p = 0
    }
    epi_sync<P::kEW>();
    float2 nl[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) nl[c] = make_float2(lse_s[col0 + 2 * c], lse_s[col0 + 2 * c + 1]);
    for (int t0 = it.ta; t0 < it.tb; t0 += kTileKeys) {
      // the tensor-memory loads below are warp-collective: decide per warp
      const bool ok = __all_sync(0xffffffffu, !aborted(flag) && mbar_wait(tfull(ts), tph));
      if (!ok && e.lane == 0) fail(a, flag, kWhereEpilogue);
      if (ok) {
        tc_fence_after();
        float v64[64];
        tmem_ld64(tmem + ((uint32_t)(e.quarter * 32) << 16) + ts * RT + col0, v64);
        tc_fence_before();
        __syncwarp();
        if (e.lane == 0) mbar_arrive(tempty(ts));
        const float red = a.sh.logits ? linmass64<MAXW>(v64, nl, heads_from(a.sh, col0))
                                       : colmass64<MAXW>(v64, nl, scale);
        const int key = t0 + e.lrow;
        if (key < it.tb) {
          // two addends per key (one per warpgroup): the result does not depend on their order
          if constexpr (MAXW == 0) atomicAdd(&Ss[key - it.ta], red);
          else max_into(&Ss[key - it.ta], red, a.sh.logits != 0);
        }
      }
      if (++ts == (int)P::kNT) { ts = 0; tph ^= 1; }
    }
    epi_sync<P::kEW>();
    if (MAXW > 0 && a.sh.logits) {   // signed group maxima: keys back to values
      for (int i = e.etid; i < it.tb - it.ta; i += kEpiThreads) Ss[i] = order_key_value(__float_as_uint(Ss[i]));
      epi_sync<P::kEW>();
    }
    if (aborted(flag)) continue;
    // max-pool over prefix positions, then page reduce (DELTA key designs 2-3)
    const SeqInfo si = t.s[it.b];   // a copy: loads once, whatever the table lives in
    float* out = a.scores + si.s_off + ((int64_t)it.layer * a.sh.h_kv + it.g) * it.L;
    float* pout = nullptr;
    if (P_ > 1) {
      const int n_pages = (it.L + P_ - 1) / P_;
      pout = a.page_scores + si.p_off + ((int64_t)it.layer * a.sh.h_kv + it.g) * n_pages;
    }
    pool_segment(Ss, it.ta, it.tb, it.a0, it.a1, pr, P_, a.sh.page_reduce, a.sh.pool_type, a.sh.gscale, out, pout,
                 e.etid, kEpiThreads);
  }
}

// Pass 2 over 256 rows with 16 epilogue warps.  The pairs of warpgroups (0, 1) and (2, 3) take
// alternate tiles: pair p the tiles this CTA takes at positions of parity p, always from TMEM stage
// p.  Within a pair, warpgroup h takes rows [128 h, 128 h + 128) (TMEM columns), read as two
// 64-column halves.  The pairs run a tile apart, so one pair's waits and loads overlap the other's
// arithmetic.  A key's two partials (one per warpgroup of the pair) meet by shared-memory atomics:
// with two addends the result does not depend on their order.
template <int RT, int D, int NK, int MAXW>
__device__ void epilogue_pass2_pairs(const TcArgs& a, const SeqTable& t, uint32_t base, uint8_t* sbase,
                                     uint32_t tmem, volatile uint32_t* flag) {
  using P = Plan<true, RT, D, NK>;
  static_assert(RT == 256 && P::kEW == 16 && P::kNT == 2, "one TMEM stage per pair of warpgroups");
  constexpr int kEpiThreads = 32 * P::kEW;
  const EpiThread e = epi_thread();
  const int pair = e.wg >> 1, half = e.wg & 1;
  const uint32_t bars = base + P::kBarOff;
  const uint32_t tfull = bars + 8u * (2 * NK + pair);
  const uint32_t tempty = bars + 8u * (2 * NK + P::kNT + pair);
  float* Ss = reinterpret_cast<float*>(sbase + P::kSsOff);
  float* lse_s = reinterpret_cast<float*>(sbase + P::kLseOff);   // logits mode: row weights
  const float2* nls = reinterpret_cast<const float2*>(lse_s + 128 * half);
  const float scale = a.sh.scale_log2;
  const bool fold = P::kFold && !a.sh.logits;                    // softmax: the accumulator holds z - lse / scale
  const uint32_t lane_base = tmem + ((uint32_t)(e.quarter * 32) << 16) + pair * RT + 128 * half;
  const int pr = (a.sh.pool_k - 1) / 2;
  const int P_ = a.sh.page_size;
  uint32_t tph = 0;
  int nt = 0;                                                    // tiles this CTA has taken so far
  Work<true> work(t);
  for (Item it; work.next(t, a.sh, it);) {
    epi_sync<P::kEW>();                                  // readers of the previous item are done
    for (int i = e.etid; i < it.tb - it.ta; i += kEpiThreads) Ss[i] = 0.f;
    for (int i = e.etid; i < RT && !fold; i += kEpiThreads) {
      const int rr = real_row(a.sh, i);
      if (a.sh.logits) lse_s[i] = rr >= 0 ? a.sh.scale_nat : 0.f;
      else lse_s[i] = rr >= 0 ? -a.lse[(int64_t)it.unit * a.sh.R + rr] : -INFINITY;
    }
    epi_sync<P::kEW>();
    for (int t0 = it.ta; t0 < it.tb; t0 += kTileKeys, ++nt) {
      if ((nt & 1) != pair) continue;
      // the tensor-memory loads below are warp-collective: decide per warp
      const bool ok = __all_sync(0xffffffffu, !aborted(flag) && mbar_wait(tfull, tph));
      tph ^= 1;
      if (!ok) {
        if (e.lane == 0) fail(a, flag, kWhereEpilogue);
        continue;
      }
      tc_fence_after();
      float r0, r1;
      {
        float v[64];
        tmem_ld64(lane_base, v);
        r0 = fold ? colmass64<MAXW, true>(v, nullptr, scale)
                  : (a.sh.logits ? linmass64<MAXW>(v, nls, heads_from(a.sh, 128 * half))
                                 : colmass64<MAXW>(v, nls, scale));
      }
      {
        float v[64];
        tmem_ld64(lane_base + 64, v);
        tc_fence_before();
        __syncwarp();
        if (e.lane == 0) mbar_arrive(tempty);
        r1 = fold ? colmass64<MAXW, true>(v, nullptr, scale)
                  : (a.sh.logits ? linmass64<MAXW>(v, nls + 32, heads_from(a.sh, 128 * half + 64))
                                 : colmass64<MAXW>(v, nls + 32, scale));
      }
      const float red = MAXW == 0 ? r0 + r1 : fmaxf(r0, r1);
      const int key = t0 + e.lrow;
      if (key < it.tb) {
        if constexpr (MAXW == 0) atomicAdd(&Ss[key - it.ta], red);
        else max_into(&Ss[key - it.ta], red, a.sh.logits != 0);
      }
    }
    epi_sync<P::kEW>();
    if (MAXW > 0 && a.sh.logits) {   // signed group maxima: keys back to values
      for (int i = e.etid; i < it.tb - it.ta; i += kEpiThreads) Ss[i] = order_key_value(__float_as_uint(Ss[i]));
      epi_sync<P::kEW>();
    }
    if (aborted(flag)) continue;
    const SeqInfo si = t.s[it.b];   // a copy: loads once, whatever the table lives in
    float* out = a.scores + si.s_off + ((int64_t)it.layer * a.sh.h_kv + it.g) * it.L;
    float* pout = nullptr;
    if (P_ > 1) {
      const int n_pages = (it.L + P_ - 1) / P_;
      pout = a.page_scores + si.p_off + ((int64_t)it.layer * a.sh.h_kv + it.g) * n_pages;
    }
    pool_segment(Ss, it.ta, it.tb, it.a0, it.a1, pr, P_, a.sh.page_reduce, a.sh.pool_type, a.sh.gscale, out, pout,
                 e.etid, kEpiThreads);
  }
}


// ---------------------------------------------------------------- kernels
template <bool PASS2, int RT, int D, int NK, int MAXW>
__global__ void __launch_bounds__(Plan<PASS2, RT, D, NK>::kThreads, 1) score_tc_kernel(const __grid_constant__ CUtensorMap tq,
                                                                 const __grid_constant__ CUtensorMap tqh,
                                                                 const __grid_constant__ CUtensorMap tk,
                                                                 const __grid_constant__ TcArgs a,
                                                                 const __grid_constant__ SeqTable tp) {
  const SeqTable& t = real_table(tp);
  {
    const Work<PASS2> mine(t);   // a grid sized for bound lengths may hold CTAs with nothing to do
    if (mine.pos >= mine.end) return;
  }
  using P = Plan<PASS2, RT, D, NK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t base = smem_addr(sbase);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sbase + P::kMiscOff);
  volatile uint32_t* flag = reinterpret_cast<volatile uint32_t*>(sbase + P::kMiscOff + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    const uint32_t bars = base + P::kBarOff;
    for (int s = 0; s < NK; ++s) {
      mbar_init(bars + 8u * s, 1);                     // full: producer arrival + TMA bytes
      mbar_init(bars + 8u * (NK + s), 1);              // empty: MMA commit
    }
    for (uint32_t s = 0; s < P::kNT; ++s) {
      mbar_init(bars + 8u * (2 * NK + s), 1);          // tfull: MMA commit
      mbar_init(bars + 8u * (2 * NK + P::kNT + s), P::kStageReaders);   // tempty: one arrival per reading warp
    }
    for (int s = 0; s < 3; ++s) mbar_init(bars + 8u * (2 * NK + 2 * P::kNT + s), 1);   // q_full, q_empty, drain
    *flag = 0;
    fence_barrier_init();
  }
  if (P::kFold && PASS2) {   // bf16 ones, the A operand of the -lse product
    uint32_t* ones = reinterpret_cast<uint32_t*>(sbase + P::kOnesOff);
    for (int i = threadIdx.x; i < 128 * 32 / 4; i += blockDim.x) ones[i] = 0x3F803F80u;
    fence_proxy_async_smem();
  }
  if (a.sh.Wp != a.sh.W) {   // padded heads: tile rows past the last head are never loaded; keep them zero
    uint4* qz = reinterpret_cast<uint4*>(sbase + P::kQOff);
    for (int i = threadIdx.x; i < (int)(P::kQBytes / 16); i += blockDim.x) qz[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(smem_addr(tslot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (warp == 0) {
    produce<PASS2, RT, D, NK>(&tq, &tqh, &tk, a, t, base, sbase, flag);
  } else if (warp == 1) {
    if (lane == 0) issue_mma<PASS2, RT, D, NK>(a, t, base, tmem, flag);
  } else {
    if constexpr (PASS2 && RT == 256) epilogue_pass2_pairs<RT, D, NK, MAXW>(a, t, base, sbase, tmem, flag);
    else if constexpr (PASS2) epilogue_pass2<RT, D, NK, MAXW>(a, t, base, sbase, tmem, flag);
    else epilogue_pass1<RT, D, NK>(a, t, base, sbase, tmem, flag);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 2-D view [rows][D] bf16, boxes of 64 x box_rows with 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, int64_t rows, int D, int box_rows = 128) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DevInfo {
  int sms = 0;
  int major = 0;
};

DevInfo device_info() {
  static std::mutex mu;
  static DevInfo cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DevInfo{};
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev].sms == 0) {
    cudaDeviceGetAttribute(&cache[dev].sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&cache[dev].major, cudaDevAttrComputeCapabilityMajor, dev);
  }
  return cache[dev];
}

template <bool PASS2, int RT, int D, int NK, int MAXW>
kvsel_status launch_one(const char* name, const CUtensorMap& tq, const CUtensorMap& tqh, const CUtensorMap& tk,
                        const TcArgs& a, const SeqTable& t, int sms, cudaStream_t s) {
  using P = Plan<PASS2, RT, D, NK>;
  auto kern = score_tc_kernel<PASS2, RT, D, NK, MAXW>;
  if (set_smem((const void*)kern, P::kSmem) != cudaSuccess) return KVSEL_ERR_CUDA;
  const int grid = t.n_items < sms ? t.n_items : sms;
  TraceScope ts(name, s);
  kern<<<grid, P::kThreads, P::kSmem, s>>>(tq, tqh, tk, a, t);
  return launch_status();
}

template <int RT, int D>
kvsel_status run_tc(const TcArgs& a, const SeqTable& t1, const SeqTable& t2, const CUtensorMap& tq,
                    const CUtensorMap& tqh, const CUtensorMap& tk, int sms, cudaStream_t s) {
  // K stages: as many as shared memory holds beside Q (and pass 2's segment buffers)
  constexpr int NK1 = (RT == 256 && D == 128) ? 5 : 4;
  constexpr int NK = (RT == 256 && D == 128) ? 3 : 4;
  kvsel_status st;
  if (!a.sh.logits && !a.sh.lse_given) {   // the softmax needs each row's log-sum-exp first
    if ((st = launch_one<false, RT, D, NK1, 0>("score_pass1_tc", tq, tqh, tk, a, t1, sms, s)) != KVSEL_OK) return st;
    if ((st = launch_lse_combine(a.sh, t1, a.part, a.lse, s)) != KVSEL_OK) return st;
  }
  if (a.sh.group_reduce != KVSEL_REDUCE_MAX)
    return launch_one<true, RT, D, NK, 0>("score_pass2_tc", tq, tqh, tk, a, t2, sms, s);
  switch (a.sh.Wp) {
    case 8: return launch_one<true, RT, D, NK, 8>("score_pass2_tc", tq, tqh, tk, a, t2, sms, s);
    case 16: return launch_one<true, RT, D, NK, 16>("score_pass2_tc", tq, tqh, tk, a, t2, sms, s);
    case 32: return launch_one<true, RT, D, NK, 32>("score_pass2_tc", tq, tqh, tk, a, t2, sms, s);
    case 64: return launch_one<true, RT, D, NK, 64>("score_pass2_tc", tq, tqh, tk, a, t2, sms, s);
  }
  return KVSEL_ERR_UNSUPPORTED;
}

}  // namespace

kvsel_status launch_score(const ScoreShape& sh_in, const SeqTable& base, const void* q, const void* k,
                          float* scores, float* page_scores, float* lse, float2* part, DeviceError* err,
                          cudaStream_t s) {
  ScoreShape sh = sh_in;
  const int64_t ups = (int64_t)sh.n_layers * sh.h_kv;
  int64_t k_rows = 0;
  for (int b = 0; b < base.batch; ++b) k_rows += ups * base.s[b].n_keys;
  const int64_t q_rows = (int64_t)base.batch * sh.n_layers * sh.h_q * sh.W;
  const DevInfo dev = device_info();
  // group max: register-resident heads of 8 .. 64 tile rows; a window that is not a power of two is
  // padded to one (the padding rows carry no mass), so the group is G Wp tile rows
  if (sh.group_reduce == KVSEL_REDUCE_MAX) {
    sh.Wp = 8;
    while (sh.Wp < sh.W) sh.Wp *= 2;
  }
  const int rows_tile = sh.G * sh.Wp;
  const bool tc = dev.major == 10 && dev.sms > 0 && rows_tile <= 256 && sh.Wp <= 64 && k_rows + 256 < (int64_t(1) << 31) &&
                  q_rows + 256 < (int64_t(1) << 31) && encode_fn() != nullptr;
  sh.seg1 = (int32_t)kScoreSeg1;
  SeqTable t1, t2;
  kvsel_status st = with_items(base, ups, kScoreSeg1, true, sh.W, 0, s, &t1);
  if (st != KVSEL_OK) return st;
  if (!tc) {
    sh.seg2 = (int32_t)(sh.page_size * ((1024 + sh.page_size - 1) / sh.page_size));
    if ((st = with_items(base, ups, sh.seg2, false, sh.W, 1, s, &t2)) != KVSEL_OK) return st;
    return launch_score_simt(sh, t1, t2, q, k, scores, page_scores, lse, part, err, s);
  }
  CUtensorMap tq, tqh, tk;
  if (!make_map(&tq, q, q_rows, sh.d) || !make_map(&tk, k, k_rows, sh.d)) return KVSEL_ERR_CUDA;
  if (sh.Wp != sh.W) {   // per-head boxes of Wp rows for the padded layout
    if (!make_map(&tqh, q, q_rows, sh.d, sh.Wp)) return KVSEL_ERR_CUDA;
  } else {
    tqh = tq;
  }
  sh.seg2 = (int32_t)(sh.page_size * (kSeg2Max / sh.page_size));
  // one item per prefix page
  if ((st = with_items(base, ups, sh.page_size, false, sh.W, 1, s, &t2)) != KVSEL_OK) return st;
  TcArgs a;
  a.sh = sh;
  a.scores = scores;
  a.page_scores = page_scores;
  a.lse = lse;
  a.part = part;
  a.err = err;
  if (rows_tile <= 128) return sh.d == 64 ? run_tc<128, 64>(a, t1, t2, tq, tqh, tk, dev.sms, s)
                                          : run_tc<128, 128>(a, t1, t2, tq, tqh, tk, dev.sms, s);
  return sh.d == 64 ? run_tc<256, 64>(a, t1, t2, tq, tqh, tk, dev.sms, s)
                    : run_tc<256, 128>(a, t1, t2, tq, tqh, tk, dev.sms, s);
}

}  // namespace kvsel
