// Top-k selection with ties to the lower index, recency / window append, and the
// aggregation of group scores across KV heads and layers (L1-normalised mean or max), pooled.
//
// Top-k: one CTA per (sequence, layer, KV head) row.  Scores map to order-
// preserving uint32 keys.  The k-th largest key T and how many keys equal to T
// are taken (krem) come from a 4-pass 8-bit radix select: over a short list of
// candidates when a sample of the row brackets the k-th key (every key at or
// above a threshold read off a 1024-key sample, some 1.25 k of them), over the
// whole row otherwise.  Then one ordered pass emits every index with key > T
// and the first krem indices with key == T, in ascending index order, which is
// exactly the first k of the ranking by (score descending, index ascending)
// sorted back into position order (DELTA, 'Key designs' 2; ClusterAttn,
// 'Method details').
#include <algorithm>

#include "internal.cuh"

namespace kvsel {
namespace {

// Threads per top-k CTA: 512 (two CTAs per SM) when the rows fit one wave of them; 256 (four per SM,
// each row's passes longer) when there are more rows than that, so that more rows run at once.
constexpr int kTopkThreadsMax = 512;
constexpr int kSmemKeysMax = 40960;   // rows up to this length are staged in shared memory

__device__ __forceinline__ uint32_t f2key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;                  // -0 ranks equal to +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the block of a 64-bit value; *total gets the block sum.
__device__ unsigned long long block_scan_u64(unsigned long long v, unsigned long long* sh32,
                                             unsigned long long* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh32[wid] = x;
  __syncthreads();
  if (wid == 0) {
    const int nw = blockDim.x >> 5;
    unsigned long long w = lane < nw ? sh32[lane] : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh32[lane] = w;
  }
  __syncthreads();
  const unsigned long long before = (wid > 0 ? sh32[wid - 1] : 0ull) + x - v;
  *total = sh32[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before;
}

struct TopkArgs {
  const float* scores;
  int32_t* idx;
  int32_t rows, k, n_recent, P, n_sel;
  int32_t stage;    // keys staged in shared memory ahead of the candidate list (0: rows read from global)
  int32_t cap;      // candidate list capacity (>= kSample), 0: no candidate path
};

constexpr int kSample = 1024;

template <int NT>
struct TopkShared {
  uint32_t hist[2][256];                     // select_short: one histogram per pass parity
  uint32_t hist_w[NT / 32][256];             // one histogram per warp: no cross-warp atomics
  unsigned long long scan_sh[32];
  uint2 warp_cnt[NT / 32];
  uint32_t sel_digit, sel_gt, n_found;
};

// The k-th largest of arr[0, n) (1 <= k <= n, a short list in shared memory): *T and how many keys
// equal to *T the top k take (*krem).  8-bit passes from the top digit; each keeps the keys that
// match the digits chosen so far, counts their next digit (one shared histogram, one atomic per key:
// on this GPU that beats grouping the lanes of equal digits by a warp match, even when every key of a
// warp has the same digit) and chooses the digit the k-th key has.  With `passes` < 4 the result
// is the k-th key's top 8 * passes bits with the rest zero: a key no larger than the k-th.  The two
// histograms alternate, so a pass zeroes the next one's while it counts into its own.
template <int NT>
__device__ void select_short(const uint32_t* arr, int n, uint32_t k, TopkShared<NT>& sh, uint32_t* T, uint32_t* krem,
                             int passes = 4) {
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t prefix = 0, pmask = 0, rem = k;
  if (tid < 256) sh.hist[0][tid] = 0;
  __syncthreads();
  for (int pass = 0; pass < passes; ++pass) {
    const int shift = 24 - 8 * pass;
    uint32_t* hist = sh.hist[pass & 1];
    if (tid < 256) sh.hist[(pass + 1) & 1][tid] = 0;
    for (int base = 0; base < n; base += NT) {
      const int i = base + tid;
      uint32_t key = 0;
      bool ok = false;
      if (i < n) {
        key = arr[i];
        ok = (key & pmask) == prefix;
      }
      if (ok) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {   // one warp: lane l holds digits 255 - 8l .. 248 - 8l, scanned from the top
      uint32_t c[8], s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        s += c[j];
      }
      uint32_t incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t above = incl - s;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (above < rem && rem <= above + c[j]) {
          sh.sel_digit = 255u - 8u * lane - j;
          sh.sel_gt = above;
        }
        above += c[j];
      }
    }
    __syncthreads();
    prefix |= sh.sel_digit << shift;
    pmask |= 255u << shift;
    rem -= sh.sel_gt;
  }
  __syncthreads();     // every thread has read sel_digit / sel_gt before they are written again
  *T = prefix;
  *krem = rem;
}

template <bool SMEM, int NT>
__global__ void __launch_bounds__(NT, 1024 / NT) topk_kernel(const __grid_constant__ TopkArgs a,
                                                            const __grid_constant__ SeqTable tp) {
  const SeqTable& t = real_table(tp);
  extern __shared__ __align__(16) uint32_t keys_sm[];   // [stage] staged keys, then [cap] candidates
  __shared__ TopkShared<NT> sh;
  uint32_t* hist = sh.hist[0];
  auto& hist_w = sh.hist_w;
  unsigned long long* scan_sh = sh.scan_sh;
  uint2* warp_cnt = sh.warp_cnt;
  uint32_t* cand = keys_sm + a.stage;

  const int row = blockIdx.x;
  const int b = row / a.rows;
  const int lg = row % a.rows;
  const SeqInfo si = t.s[b];   // a copy: loads once, whatever the table lives in
  if (si.L == 0) return;                 // a table whose device lengths failed the checks
  const int n = a.P == 1 ? si.L : (si.L + a.P - 1) / a.P;
  const int n_cand = n - a.n_recent;
  const float* src = a.scores + (a.P == 1 ? si.s_off : si.p_off) + (int64_t)lg * n;
  int32_t* out = a.idx + (int64_t)row * a.n_sel;
  const int tid = threadIdx.x;

  if (SMEM) {
    // stage the row's keys: 16-byte loads when the row is 16-byte aligned, several in flight per thread
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
      const int n4 = n_cand >> 2;
      const float4* s4 = reinterpret_cast<const float4*>(src);
      uint4* k4 = reinterpret_cast<uint4*>(keys_sm);
#pragma unroll 4
      for (int i = tid; i < n4; i += NT) {
        const float4 f = s4[i];
        k4[i] = make_uint4(f2key(f.x), f2key(f.y), f2key(f.z), f2key(f.w));
      }
      for (int i = 4 * n4 + tid; i < n_cand; i += NT) keys_sm[i] = f2key(src[i]);
    } else {
#pragma unroll 8
      for (int i = tid; i < n_cand; i += NT) keys_sm[i] = f2key(src[i]);
    }
  }
  __syncthreads();
  auto key_at = [&](int i) -> uint32_t { return SMEM ? keys_sm[i] : f2key(src[i]); };

  uint32_t prefix = 0, pmask = 0;
  uint32_t krem = (uint32_t)a.k;
  bool have = false;   // T (prefix) and krem found from the candidate list
  int n_list = -1;     // >= 0: the list holds every candidate in index order and the emission walks it
  const int lane = tid & 31, warp = tid >> 5;
  const unsigned lower = (1u << lane) - 1u;
  constexpr int kWarps = NT / 32;
  if (a.k > 0 && a.cap >= kSample && n_cand >= (SMEM ? 12 : 4) * kSample) {
    // A threshold read off an evenly spaced sample: about k * S / n_cand sample keys lie at or above the
    // row's k-th key; the sample's r0-th largest key, r0 1.25 times that plus three standard deviations,
    // leaves some 1.25 k keys of the row at or above it, the k-th among them.  Its top 16 bits suffice
    // (two passes): the threshold is then a little lower, and the list a little longer.
    const float e = (float)a.k * (float)kSample / (float)n_cand;
    const int r0 = (int)(1.25f * e + 3.0f * sqrtf(e) + 4.0f);
    if (r0 <= kSample) {
      for (int s = tid; s < kSample; s += NT) cand[s] = key_at((int)(((int64_t)s * n_cand) / kSample));
      __syncthreads();
      uint32_t T0, rem0;
      select_short(cand, kSample, (uint32_t)r0, sh, &T0, &rem0, 2);
      if (!SMEM) {
        // Rows read from memory: every key >= T0 into the list in index order.  Each warp counts its
        // contiguous segment's candidates, the counts give each warp its place, and a second read of
        // the segment (now in L2) writes the keys and their positions.  The segments are runs of
        // 16-byte units of the row (the keys before the first 16-byte boundary go to warp 0, the last
        // 0-3 keys to the last warp), four keys per lane and load.
        const int head = min(n_cand, (int)((4u - (uint32_t)((reinterpret_cast<uintptr_t>(src) >> 2) & 3u)) & 3u));
        const int m4 = (n_cand - head) >> 2;
        const int tail0 = head + 4 * m4;
        const float4* s4 = reinterpret_cast<const float4*>(src + head);
        const int u0 = (int)(((int64_t)warp * m4) / kWarps), u1 = (int)(((int64_t)(warp + 1) * m4) / kWarps);
        uint32_t c = 0;
        if (warp == 0 && lane < head) c += f2key(src[lane]) >= T0 ? 1u : 0u;
        if (warp == kWarps - 1 && lane < n_cand - tail0) c += f2key(src[tail0 + lane]) >= T0 ? 1u : 0u;
#pragma unroll 4
        for (int u = u0 + lane; u < u1; u += 32) {
          const float4 f = s4[u];
          c += (f2key(f.x) >= T0 ? 1u : 0u) + (f2key(f.y) >= T0 ? 1u : 0u) + (f2key(f.z) >= T0 ? 1u : 0u) +
               (f2key(f.w) >= T0 ? 1u : 0u);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        if (lane == 0) warp_cnt[warp] = make_uint2(c, 0u);
        __syncthreads();
        uint32_t pos = 0, nf = 0;
        for (int w = 0; w < kWarps; ++w) {
          if (w < warp) pos += warp_cnt[w].x;
          nf += warp_cnt[w].x;
        }
        if (nf >= (uint32_t)a.k && nf <= (uint32_t)a.cap) {   // the row's k-th key is among them
          uint32_t* cand_idx = cand + a.cap;
          auto put1 = [&](bool live, int i) {     // one key per lane, lanes in index order
            const uint32_t key = live ? f2key(src[i]) : 0u;
            const bool p = live && key >= T0;
            const unsigned m = __ballot_sync(0xffffffffu, p);
            if (p) {
              const uint32_t at = pos + (uint32_t)__popc(m & lower);
              cand[at] = key;
              cand_idx[at] = (uint32_t)i;
            }
            pos += (uint32_t)__popc(m);
          };
          if (warp == 0) put1(lane < head, lane);
          constexpr int U = 4;                 // rounds of 32 units whose loads are issued together
          for (int base = u0; base < u1; base += 32 * U) {
            float4 f[U];
#pragma unroll
            for (int r = 0; r < U; ++r) {
              const int u = base + 32 * r + lane;
              f[r] = u < u1 ? s4[u] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int r = 0; r < U; ++r) {
              const int u = base + 32 * r + lane;
              const bool live = u < u1;
              const uint32_t kk[4] = {f2key(f[r].x), f2key(f[r].y), f2key(f[r].z), f2key(f[r].w)};
              bool p[4];
              uint32_t before = 0, all = 0;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                p[q] = live && kk[q] >= T0;
                const unsigned m = __ballot_sync(0xffffffffu, p[q]);
                before += (uint32_t)__popc(m & lower);
                all += (uint32_t)__popc(m);
              }
              // the lane's four keys follow every key of the lanes before it
              uint32_t at = pos + before;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                if (p[q]) {
                  cand[at] = kk[q];
                  cand_idx[at] = (uint32_t)(head + 4 * u + q);
                  ++at;
                }
              }
              pos += all;
            }
          }
          if (warp == kWarps - 1) put1(lane < n_cand - tail0, tail0 + lane);
          __syncthreads();
          select_short(cand, (int)nf, (uint32_t)a.k, sh, &prefix, &krem);
          n_list = (int)nf;
          have = true;
        }
      } else {
        if (tid == 0) sh.n_found = 0;
        __syncthreads();
        // staged rows: every key >= T0 into the list (positions taken a warp at a time); keys past the
        // capacity are counted but not stored, and the list is then not used
#pragma unroll 4
        for (int base = 0; base < n_cand; base += NT) {
          const int i = base + tid;
          const uint32_t key = i < n_cand ? key_at(i) : 0u;
          const bool p = i < n_cand && key >= T0;
          const unsigned m = __ballot_sync(0xffffffffu, p);
          uint32_t wbase = 0;
          if (lane == 0 && m != 0u) wbase = atomicAdd(&sh.n_found, (uint32_t)__popc(m));
          wbase = __shfl_sync(0xffffffffu, wbase, 0);
          const uint32_t at = wbase + (uint32_t)__popc(m & lower);
          if (p && at < (uint32_t)a.cap) cand[at] = key;
        }
        __syncthreads();
        const uint32_t nf = sh.n_found;
        if (nf >= (uint32_t)a.k && nf <= (uint32_t)a.cap) {   // the row's k-th key is among them
          select_short(cand, (int)nf, (uint32_t)a.k, sh, &prefix, &krem);
          have = true;
        }
      }
    }
  }
  if (a.k > 0) {
    for (int pass = 0; !have && pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      uint32_t* hw = hist_w[tid >> 5];
      for (int j = tid & 31; j < 256; j += 32) hw[j] = 0;
      __syncwarp();
#pragma unroll 4
      for (int base = 0; base < n_cand; base += NT) {
        const int i = base + tid;
        uint32_t key = 0;
        bool ok = false;
        if (i < n_cand) {
          key = key_at(i);
          ok = (key & pmask) == prefix;
        }
        if (ok) atomicAdd(&hw[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid < 256) {
        uint32_t c = 0;
#pragma unroll 8
        for (int w = 0; w < NT / 32; ++w) c += hist_w[w][tid];
        hist[tid] = c;
      }
      __syncthreads();
      // digits from the top: count of candidates whose digit is above d
      const uint32_t d = 255u - (uint32_t)tid;
      const unsigned long long c = tid < 256 ? hist[d] : 0ull;
      unsigned long long tot;
      const unsigned long long above = block_scan_u64(c, scan_sh, &tot);
      if (tid < 256 && above < krem && krem <= above + c) {
        sh.sel_digit = d;
        sh.sel_gt = (uint32_t)above;
      }
      __syncthreads();
      prefix |= sh.sel_digit << shift;
      pmask |= 255u << shift;
      krem -= sh.sel_gt;
      __syncthreads();
    }
    // ordered emission: every key > T and the first krem keys == T, in index order.  A selected key's
    // output position is the number of selected keys before it: (keys > T before it) + min(keys == T
    // before it, krem).  Each warp owns one contiguous segment (of the row, or of the candidate list,
    // which is in index order): it counts its segment's keys > T and == T, one barrier makes every
    // warp's counts visible, and the warp then walks its segment in rounds of 32 consecutive keys,
    // placing each key from its warp's offsets and the ballots of the lanes before it.
    const uint32_t T = prefix;
    const uint32_t* cand_idx = cand + a.cap;
    const bool from_list = n_list >= 0;
    const int n_em = from_list ? n_list : n_cand;
    auto em_key = [&](int i) -> uint32_t { return from_list ? cand[i] : key_at(i); };
    auto em_idx = [&](int i) -> int32_t { return from_list ? (int32_t)cand_idx[i] : i; };
    const int seg = (n_em + kWarps - 1) / kWarps;
    const int s0 = min(n_em, warp * seg), s1 = min(n_em, s0 + seg);
    uint32_t g = 0, e = 0;
#pragma unroll 8
    for (int i = s0 + lane; i < s1; i += 32) {
      const uint32_t key = em_key(i);
      g += key > T ? 1u : 0u;
      e += key == T ? 1u : 0u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xffffffffu, g, o);
      e += __shfl_xor_sync(0xffffffffu, e, o);
    }
    __syncthreads();                       // (warp_cnt may still be read by the list's placement)
    if (lane == 0) warp_cnt[warp] = make_uint2(g, e);
    __syncthreads();
    uint32_t gt_before = 0, eq_before = 0;
    for (int w = 0; w < warp; ++w) {
      gt_before += warp_cnt[w].x;
      eq_before += warp_cnt[w].y;
    }
    constexpr int U = 4;                       // rounds whose loads are issued together
    for (int base = s0; base < s1; base += 32 * U) {
      uint32_t keys[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = base + 32 * u + lane;
        keys[u] = i < s1 ? em_key(i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = base + 32 * u + lane;
        const bool is_gt = i < s1 && keys[u] > T;
        const bool is_eq = i < s1 && keys[u] == T;
        const unsigned mg = __ballot_sync(0xffffffffu, is_gt), me = __ballot_sync(0xffffffffu, is_eq);
        const uint32_t gb = gt_before + __popc(mg & lower), eb = eq_before + __popc(me & lower);
        if (is_gt) out[gb + min(eb, krem)] = em_idx(i);
        else if (is_eq && eb < krem) out[gb + eb] = em_idx(i);
        gt_before += __popc(mg);
        eq_before += __popc(me);
      }
    }
  }
  // recency pages, then (when appended) window pages or window tokens: the indices from n_cand on
  for (int i = tid; i < a.n_sel - a.k; i += NT) out[a.k + i] = n_cand + i;
}

// ------------------------------------------------------------------------ aggregation
constexpr int kCombThreads = 256;
// Tokens per pooling CTA: about one per thread when every token reads many layers (so that they are
// read by many threads at once), four per thread when each token reads one layer's heads.
constexpr int kCombChunkLayers = 256;
constexpr int kCombChunkMax = 1024;

struct AggArgs {
  const float* scores;      // raw group scores, per sequence [n_layers][h_kv][L]
  float* norms;             // [batch][hi - lo + 1][n_h] L1 norms (L1 mean only)
  float* out;               // per sequence [n_l][n_h][L]
  int32_t n_layers, h_kv, lo, hi, layer_op, head_op, n_l, n_h, pool_k, pool_type;
  int32_t chunk;            // tokens per pooling CTA (kCombChunkLayers or kCombChunkMax)
};

// Value of (layer, output head oh) at token tt: one KV head, or the sum over all of them.
__device__ __forceinline__ float head_value(const AggArgs& a, const SeqInfo& si, int layer, int oh, int tt) {
  const float* base = a.scores + si.s_off + (int64_t)layer * a.h_kv * si.L + tt;
  if (a.head_op == KVSEL_HEADS_EACH) return base[(int64_t)oh * si.L];
  // heads in batches of 8 whose loads are all issued before they are added, in head order
  float acc = 0.f;
  for (int g0 = 0; g0 < a.h_kv; g0 += 8) {
    float x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) x[u] = g0 + u < a.h_kv ? base[(int64_t)(g0 + u) * si.L] : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (g0 + u < a.h_kv) acc += x[u];
  }
  return acc;
}

// L1 norm over the prefix of each (sequence, layer of the range, output head) row.
__global__ void __launch_bounds__(kCombThreads) agg_norms(const __grid_constant__ AggArgs a,
                                                          const __grid_constant__ SeqTable tp) {
  const SeqTable& t = real_table(tp);
  __shared__ float red[kCombThreads];
  const int nr = a.hi - a.lo + 1;
  const int row = blockIdx.x;                        // (b, layer - lo, oh)
  const int b = row / (nr * a.n_h);
  const int rem = row % (nr * a.n_h);
  const int layer = a.lo + rem / a.n_h, oh = rem % a.n_h;
  const SeqInfo si = t.s[b];   // a copy: loads once, whatever the table lives in
  float acc = 0.f;
  for (int i = threadIdx.x; i < si.L; i += kCombThreads) acc += fabsf(head_value(a, si, layer, oh, i));
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = kCombThreads / 2; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) a.norms[row] = red[0];
}

// One chunk of one output row: the aggregated value of every token of the chunk and its pooling
// halo, then the pooled outputs of the chunk.
__global__ void __launch_bounds__(kCombThreads) agg_pool(const __grid_constant__ AggArgs a,
                                                         const __grid_constant__ SeqTable tp) {
  const SeqTable& t = real_table(tp);
  __shared__ float S[kCombChunkMax + 64];
  const int b = blockIdx.z;
  const int ol = blockIdx.y / a.n_h, oh = blockIdx.y % a.n_h;
  const SeqInfo si = t.s[b];   // a copy: loads once, whatever the table lives in
  const int a0 = blockIdx.x * a.chunk;
  if (a0 >= si.L) return;
  const int a1 = min(si.L, a0 + a.chunk);
  const int pr = (a.pool_k - 1) / 2;
  const int ea = max(0, a0 - pr), eb = min(si.L, a1 + pr);
  const int nr = a.hi - a.lo + 1;
  const float inv_n = 1.0f / (float)nr;
  for (int tt = ea + threadIdx.x; tt < eb; tt += kCombThreads) {
    float v;
    if (a.layer_op == KVSEL_LAYERS_EACH) {
      v = head_value(a, si, a.lo + ol, oh, tt);
    } else {
      // layers in batches of 16 whose loads are all issued before they are combined, in layer order
      // (the same arithmetic, in the same order, as one layer at a time)
      const bool mx = a.layer_op == KVSEL_LAYERS_MAX;
      float acc = mx ? -INFINITY : 0.f;
      for (int l0 = a.lo; l0 <= a.hi; l0 += 16) {
        float x[16], nv[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int layer = l0 + u;
          x[u] = 0.f;
          nv[u] = 1.f;
          if (layer <= a.hi) {
            x[u] = head_value(a, si, layer, oh, tt);
            if (!mx) nv[u] = a.norms[((int64_t)b * nr + (layer - a.lo)) * a.n_h + oh];
          }
        }
#pragma unroll
        for (int u = 0; u < 16; ++u)
          if (l0 + u <= a.hi) acc = mx ? fmaxf(acc, x[u]) : acc + x[u] / nv[u];
      }
      v = mx ? acc : acc * inv_n;
    }
    S[tt - ea] = v;
  }
  __syncthreads();
  const int64_t tok_off = si.s_off / ((int64_t)a.n_layers * a.h_kv);   // tokens of earlier sequences
  float* out = a.out + tok_off * a.n_l * a.n_h + ((int64_t)ol * a.n_h + oh) * si.L;
  for (int tt = a0 + threadIdx.x; tt < a1; tt += kCombThreads) {
    const int l0 = max(tt - pr, ea), l1 = min(tt + pr, eb - 1);
    float u = S[l0 - ea];
    if (a.pool_type == KVSEL_POOL_AVG) {
      for (int x = l0 + 1; x <= l1; ++x) u += S[x - ea];
      u /= (float)(l1 - l0 + 1);
    } else {
      for (int x = l0 + 1; x <= l1; ++x) u = fmaxf(u, S[x - ea]);
    }
    out[tt] = u;
  }
}

}  // namespace

kvsel_status launch_topk(const kvsel_desc& d, const SeqTable& t, int rows, int k, int n_recent,
                         bool append_window, const float* scores, int32_t* idx, cudaStream_t s) {
  TopkArgs a;
  a.scores = scores;
  a.idx = idx;
  a.rows = rows;
  a.k = k;
  a.n_recent = n_recent;
  a.P = d.page_size;
  a.n_sel = d.page_size == 1 ? k + (append_window ? d.window : 0)
                             : k + n_recent + (append_window ? d.window / d.page_size : 0);
  int64_t nmax = 0;   // from the host table: the real lengths, or their bound with device lengths
  for (int b = 0; b < d.batch; ++b) {
    const int64_t L = t.s[b].L;
    const int64_t n = d.page_size == 1 ? L : (L + d.page_size - 1) / d.page_size;
    nmax = n > nmax ? n : nmax;
  }
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return KVSEL_ERR_CUDA;
  // rows of 12K keys or more are read from memory and take the ordered candidate list (keys and
  // positions); shorter rows are staged in shared memory
  const bool staged = nmax < 12 * kSample && nmax <= kSmemKeysMax;
  a.stage = staged ? (int32_t)nmax : 0;
  // candidate list: room for 2 k + 2048 entries (the sample's threshold keeps ~1.25 k; more than 2 k + 2048
  // is several standard deviations out, and then the whole-row select runs) within what shared memory
  // has left beside the staged row and the kernel's own arrays
  const int64_t entry = staged ? 1 : 2;      // a key, or a key and its position
  const int64_t avail = (((int64_t)optin - (int64_t)sizeof(TopkShared<kTopkThreadsMax>) - 256) / 4 - a.stage) / entry;
  const int64_t cap = std::min<int64_t>(std::max<int64_t>(kSample, 2 * (int64_t)k + 2048), avail);
  a.cap = cap >= kSample ? (int32_t)cap : 0;
  const size_t smem = (size_t)(a.stage + entry * a.cap) * sizeof(uint32_t);
  const int grid = d.batch * rows;
  // more rows than one wave of 512-thread CTAs (two per SM): 256-thread CTAs, four per SM
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KVSEL_ERR_CUDA;
  const bool many = grid > 2 * sms;
  TraceScope ts("topk_radix", s);
  if (staged) {
    if (many) {
      if (set_smem((const void*)topk_kernel<true, 256>, smem) != cudaSuccess) return KVSEL_ERR_CUDA;
      topk_kernel<true, 256><<<grid, 256, smem, s>>>(a, t);
    } else {
      if (set_smem((const void*)topk_kernel<true, 512>, smem) != cudaSuccess) return KVSEL_ERR_CUDA;
      topk_kernel<true, 512><<<grid, 512, smem, s>>>(a, t);
    }
  } else {
    if (many) {
      if (set_smem((const void*)topk_kernel<false, 256>, smem) != cudaSuccess) return KVSEL_ERR_CUDA;
      topk_kernel<false, 256><<<grid, 256, smem, s>>>(a, t);
    } else {
      if (set_smem((const void*)topk_kernel<false, 512>, smem) != cudaSuccess) return KVSEL_ERR_CUDA;
      topk_kernel<false, 512><<<grid, 512, smem, s>>>(a, t);
    }
  }
  return launch_status();
}

kvsel_status launch_aggregate(const kvsel_desc& d, const SeqTable& t, const float* scores, int lo, int hi,
                              int layer_op, int head_op, float* norms, float* out, cudaStream_t s) {
  AggArgs a;
  a.scores = scores;
  a.norms = norms;
  a.out = out;
  a.n_layers = d.n_layers;
  a.h_kv = d.h_kv;
  a.lo = lo;
  a.hi = hi;
  a.layer_op = layer_op;
  a.head_op = head_op;
  a.n_l = layer_op == KVSEL_LAYERS_EACH ? hi - lo + 1 : 1;
  a.n_h = head_op == KVSEL_HEADS_EACH ? d.h_kv : 1;
  a.pool_k = d.pool_k;
  a.pool_type = d.pool_type;
  kvsel_status st;
  if (layer_op == KVSEL_LAYERS_L1_MEAN) {
    TraceScope ts("layer_norms", s);
    agg_norms<<<d.batch * (hi - lo + 1) * a.n_h, kCombThreads, 0, s>>>(a, t);
    if ((st = launch_status()) != KVSEL_OK) return st;
  }
  int64_t lmax = 0;   // real lengths, or their bound with device lengths
  for (int b = 0; b < d.batch; ++b) lmax = t.s[b].L > lmax ? t.s[b].L : lmax;
  a.chunk = layer_op == KVSEL_LAYERS_EACH ? kCombChunkMax : kCombChunkLayers;
  dim3 grid((unsigned)((lmax + a.chunk - 1) / a.chunk), (unsigned)(a.n_l * a.n_h), d.batch);
  TraceScope ts("aggregate_pool", s);
  agg_pool<<<grid, kCombThreads, 0, s>>>(a, t);
  return launch_status();
}

}  // namespace kvsel
