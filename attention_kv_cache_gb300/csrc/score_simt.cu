// Window-attention scoring on CUDA cores (fp32 FMA), two passes over the keys.
//
// ClusterAttn, 'Background and key observations': the window queries' logits
// against every prompt key, a causal mask inside the window, a softmax over
// the full row, and the column sum over the window rows for prefix columns.
// The softmax needs each row's log-sum-exp over all its keys before any
// column can be summed, so:
//   pass 1  — per (unit, key segment): online max / sum of 2^(z - m) per row
//   combine — per row: lse = M + log2(sum_s l_s 2^(m_s - M))
//   pass 2  — per (unit, prefix segment): p = 2^(z - lse), column mass per
//             head, group sum / max / mean, max or average pool (halo keys
//             recomputed), page reduce.
// Logits are never stored.  Exponentials are base 2 on z * log2(e)/sqrt(d).
// In logits mode (GemFilter's pre-softmax scores) pass 2 alone runs and sums
// z / sqrt(d) over the window rows instead of probabilities.
#include "internal.cuh"

namespace kvsel {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 32;   // keys per tile

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct ScoreArgs {
  ScoreShape sh;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  float* scores;
  float* page_scores;
  float* lse;
  float2* part;
  DeviceError* err;
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Window queries of unit (b, layer, g) as fp32 rows r = h_local * W + j; rows >= R are zero.
template <int D, int RP>
__device__ void load_q(float* Qs, const ScoreArgs& a, int b, int layer, int g) {
  constexpr int LD = D + 4;
  const ScoreShape& sh = a.sh;
  for (int v = threadIdx.x; v < RP * (D / 8); v += kThreads) {
    const int r = v / (D / 8), c8 = (v % (D / 8)) * 8;
    float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (r < sh.R) {
      const int h = g * sh.G + r / sh.W, j = r % sh.W;
      const int64_t off = ((((int64_t)b * sh.n_layers + layer) * sh.h_q + h) * sh.W + j) * D + c8;
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(a.q + off), f);
    }
    float4* dst = reinterpret_cast<float4*>(Qs + r * LD + c8);
    dst[0] = make_float4(f[0], f[1], f[2], f[3]);
    dst[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
}

// Keys t0 .. t0 + kTile - 1 of one unit (rows from kbase); keys >= tend load as zero.
template <int D>
__device__ void load_k_tile(float* Ks, const __nv_bfloat16* kbase, int t0, int tend) {
  constexpr int LD = D + 4;
  for (int v = threadIdx.x; v < kTile * (D / 8); v += kThreads) {
    const int i = v / (D / 8), c8 = (v % (D / 8)) * 8;
    float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (t0 + i < tend) bf16x8_to_f32(*reinterpret_cast<const uint4*>(kbase + (int64_t)(t0 + i) * D + c8), f);
    float4* dst = reinterpret_cast<float4*>(Ks + i * LD + c8);
    dst[0] = make_float4(f[0], f[1], f[2], f[3]);
    dst[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
}

// acc[i] = <q_r, k_{s + i * TPR}> for the KPT keys of this thread.
template <int D, int KPT>
__device__ __forceinline__ void tile_dots(const float* Qs, const float* Ks, int r, int s, float* acc) {
  constexpr int LD = D + 4;
  constexpr int TPR = kTile / KPT;
#pragma unroll
  for (int i = 0; i < KPT; ++i) acc[i] = 0.f;
#pragma unroll 4
  for (int c = 0; c < D; c += 4) {
    const float4 qv = *reinterpret_cast<const float4*>(Qs + r * LD + c);
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      const float4 kv = *reinterpret_cast<const float4*>(Ks + (s + i * TPR) * LD + c);
      acc[i] = fmaf(qv.x, kv.x, acc[i]);
      acc[i] = fmaf(qv.y, kv.y, acc[i]);
      acc[i] = fmaf(qv.z, kv.z, acc[i]);
      acc[i] = fmaf(qv.w, kv.w, acc[i]);
    }
  }
}

__device__ __forceinline__ const __nv_bfloat16* unit_keys(const ScoreArgs& a, const SeqInfo& si, int layer, int g) {
  return a.k + si.k_off + ((int64_t)layer * a.sh.h_kv + g) * si.n_keys * a.sh.d;
}

// ------------------------------------------------------------------------ pass 1
template <int D, int RP>
__global__ void __launch_bounds__(kThreads) score_pass1_simt(const __grid_constant__ ScoreArgs a,
                                                             const __grid_constant__ SeqTable tp) {
  const SeqTable& t = real_table(tp);
  constexpr int KPT = RP / 8, TPR = kTile / KPT, LD = D + 4;
  extern __shared__ __align__(16) float smem[];
  float* Qs = smem;
  float* Ks = Qs + RP * LD;
  float* red_m = Ks + kTile * LD;
  float* red_l = red_m + kThreads;

  const ScoreShape& sh = a.sh;
  const int item = blockIdx.x;
  if (item >= t.n_items) return;         // the grid is sized for bound lengths
  const int b = find_seq(t, item);
  const SeqInfo si = t.s[b];   // a copy: loads once, whatever the table lives in
  const int local = item - si.item0;
  const int ul = local / si.n_seg, seg = local % si.n_seg;
  const int layer = ul / sh.h_kv, g = ul % sh.h_kv;
  const int ta = seg * sh.seg1;
  const int tb = min(si.n_keys, ta + sh.seg1);
  const __nv_bfloat16* kb = unit_keys(a, si, layer, g);

  load_q<D, RP>(Qs, a, b, layer, g);
  const int r = threadIdx.x % RP, s = threadIdx.x / RP;
  const bool rvalid = r < sh.R;
  const int row_last = si.L + (rvalid ? r % sh.W : 0);   // last key this row sees
  float m = -INFINITY, l = 0.f;
  float acc[KPT];
  for (int t0 = ta; t0 < tb; t0 += kTile) {
    __syncthreads();
    load_k_tile<D>(Ks, kb, t0, tb);
    __syncthreads();
    tile_dots<D, KPT>(Qs, Ks, r, s, acc);
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      const int key = t0 + s + i * TPR;
      if (rvalid && key < tb && key <= row_last) mx = fmaxf(mx, acc[i] * sh.scale_log2);
    }
    if (mx > -INFINITY) {
      const float nm = fmaxf(m, mx);
      l *= fast_ex2(m - nm);
#pragma unroll
      for (int i = 0; i < KPT; ++i) {
        const int key = t0 + s + i * TPR;
        if (key < tb && key <= row_last) l += fast_ex2(acc[i] * sh.scale_log2 - nm);
      }
      m = nm;
    }
  }
  red_m[r * TPR + s] = m;
  red_l[r * TPR + s] = l;
  __syncthreads();
  if (s == 0 && rvalid) {
    float M = -INFINITY;
    for (int i = 0; i < TPR; ++i) M = fmaxf(M, red_m[r * TPR + i]);
    float S = 0.f;
    if (M > -INFINITY)
      for (int i = 0; i < TPR; ++i) {
        const float mi = red_m[r * TPR + i];
        if (mi > -INFINITY) S += red_l[r * TPR + i] * fast_ex2(mi - M);
      }
    a.part[(int64_t)item * sh.R + r] = make_float2(M, S);
  }
}

// ------------------------------------------------------------------------ combine
__global__ void __launch_bounds__(kThreads) score_lse_combine(const __grid_constant__ ScoreArgs a,
                                                              const __grid_constant__ SeqTable tp,
                                                              int64_t n_rows) {
  const SeqTable& t = real_table(tp);
  const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (i >= n_rows) return;
  const ScoreShape& sh = a.sh;
  const int64_t u = i / sh.R;
  const int r = (int)(i % sh.R);
  const int64_t ups = (int64_t)sh.n_layers * sh.h_kv;
  const int b = (int)(u / ups);
  const int ul = (int)(u % ups);
  const SeqInfo si = t.s[b];   // a copy: loads once, whatever the table lives in
  const int64_t first = si.item0 + (int64_t)ul * si.n_seg;
  float M = -INFINITY;
  for (int sg = 0; sg < si.n_seg; ++sg) M = fmaxf(M, a.part[(first + sg) * sh.R + r].x);
  float S = 0.f;
  for (int sg = 0; sg < si.n_seg; ++sg) {
    const float2 p = a.part[(first + sg) * sh.R + r];
    if (p.x > -INFINITY) S += p.y * exp2f(p.x - M);
  }
  a.lse[i] = M + log2f(S);
}

// ------------------------------------------------------------------------ pass 2
template <int D, int RP>
__global__ void __launch_bounds__(kThreads) score_pass2_simt(const __grid_constant__ ScoreArgs a,
                                                             const __grid_constant__ SeqTable tp) {
  const SeqTable& t = real_table(tp);
  constexpr int KPT = RP / 8, TPR = kTile / KPT, LD = D + 4, LDP = kTile + 1;
  extern __shared__ __align__(16) float smem[];
  const ScoreShape& sh = a.sh;
  float* Qs = smem;
  float* Ks = Qs + RP * LD;
  float* Ps = Ks + kTile * LD;
  float* Ss = Ps + RP * LDP;            // group scores of [ea, eb)
  float* Us = Ss + sh.seg2 + 128;       // pooled scores of [a0, a1)

  const int item = blockIdx.x;
  if (item >= t.n_items) return;         // the grid is sized for bound lengths
  const int b = find_seq(t, item);
  const SeqInfo si = t.s[b];   // a copy: loads once, whatever the table lives in
  const int local = item - si.item0;
  const int ul = local / si.n_seg, seg = local % si.n_seg;
  const int layer = ul / sh.h_kv, g = ul % sh.h_kv;
  const int pr = (sh.pool_k - 1) / 2;
  const int a0 = seg * sh.seg2, a1 = min(si.L, a0 + sh.seg2);
  const int ea = max(0, a0 - pr), eb = min(si.L, a1 + pr);
  const __nv_bfloat16* kb = unit_keys(a, si, layer, g);

  load_q<D, RP>(Qs, a, b, layer, g);
  const int r = threadIdx.x % RP, s = threadIdx.x / RP;
  const bool rvalid = r < sh.R;
  const float lse_r = (rvalid && !sh.logits) ? a.lse[(int64_t)(si.unit0 + ul) * sh.R + r] : 0.f;
  float acc[KPT];
  for (int t0 = ea; t0 < eb; t0 += kTile) {
    __syncthreads();
    load_k_tile<D>(Ks, kb, t0, eb);
    __syncthreads();
    tile_dots<D, KPT>(Qs, Ks, r, s, acc);
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      const int tl = s + i * TPR;
      // prefix keys are visible to every window row
      float p = 0.f;
      if (rvalid && t0 + tl < eb) p = sh.logits ? acc[i] * sh.scale_nat : fast_ex2(acc[i] * sh.scale_log2 - lse_r);
      Ps[r * LDP + tl] = p;
    }
    __syncthreads();
    if (threadIdx.x < kTile && t0 + (int)threadIdx.x < eb) {
      float red = 0.f;
      for (int h = 0; h < sh.G; ++h) {
        float cs = 0.f;
        for (int j = 0; j < sh.W; ++j) cs += Ps[(h * sh.W + j) * LDP + threadIdx.x];
        red = (h == 0) ? cs : (sh.group_reduce == KVSEL_REDUCE_MAX ? fmaxf(red, cs) : red + cs);
      }
      Ss[t0 + threadIdx.x - ea] = red;
    }
  }
  __syncthreads();
  float* out = a.scores + si.s_off + ((int64_t)layer * sh.h_kv + g) * si.L;
  for (int tt = a0 + threadIdx.x; tt < a1; tt += kThreads) {
    const int lo = max(tt - pr, ea), hi = min(tt + pr, eb - 1);
    float u = Ss[lo - ea];
    if (sh.pool_type == KVSEL_POOL_AVG) {
      for (int x = lo + 1; x <= hi; ++x) u += Ss[x - ea];
      u /= (float)(hi - lo + 1);
    } else {
      for (int x = lo + 1; x <= hi; ++x) u = fmaxf(u, Ss[x - ea]);
    }
    u *= sh.gscale;
    out[tt] = u;
    Us[tt - a0] = u;
  }
  if (sh.page_size > 1) {
    __syncthreads();
    const int P = sh.page_size;
    const int n_pages = (si.L + P - 1) / P;
    float* pout = a.page_scores + si.p_off + ((int64_t)layer * sh.h_kv + g) * n_pages;
    for (int p = a0 / P + threadIdx.x; p * P < a1; p += kThreads) {
      const int lo = p * P, hi = min(a1, lo + P);
      float v = Us[lo - a0];
      for (int x = lo + 1; x < hi; ++x)
        v = (sh.page_reduce == KVSEL_REDUCE_MAX) ? fmaxf(v, Us[x - a0]) : v + Us[x - a0];
      pout[p] = v;
    }
  }
}

template <int D, int RP>
kvsel_status run(const ScoreArgs& args, const SeqTable& t1, const SeqTable& t2, cudaStream_t s) {
  constexpr int LD = D + 4;
  const size_t smem1 = sizeof(float) * ((size_t)RP * LD + kTile * LD + 2 * kThreads);
  const size_t smem2 = sizeof(float) * ((size_t)RP * LD + kTile * LD + (size_t)RP * (kTile + 1) +
                                        2 * (size_t)args.sh.seg2 + 128);
  if (set_smem((const void*)score_pass1_simt<D, RP>, smem1) != cudaSuccess) return KVSEL_ERR_CUDA;
  if (set_smem((const void*)score_pass2_simt<D, RP>, smem2) != cudaSuccess) return KVSEL_ERR_CUDA;
  kvsel_status st;
  if (!args.sh.logits && !args.sh.lse_given) {   // the softmax needs each row's log-sum-exp first
    {
      TraceScope ts("score_pass1_simt", s);
      score_pass1_simt<D, RP><<<t1.n_items, kThreads, smem1, s>>>(args, t1);
      if ((st = launch_status()) != KVSEL_OK) return st;
    }
    const int64_t units = (int64_t)t1.batch * args.sh.n_layers * args.sh.h_kv;
    const int64_t n_rows = units * args.sh.R;
    TraceScope ts("score_lse_combine", s);
    score_lse_combine<<<(unsigned)((n_rows + kThreads - 1) / kThreads), kThreads, 0, s>>>(args, t1, n_rows);
    if ((st = launch_status()) != KVSEL_OK) return st;
  }
  {
    TraceScope ts("score_pass2_simt", s);
    score_pass2_simt<D, RP><<<t2.n_items, kThreads, smem2, s>>>(args, t2);
    if ((st = launch_status()) != KVSEL_OK) return st;
  }
  return KVSEL_OK;
}

template <int D>
kvsel_status run_d(const ScoreArgs& args, const SeqTable& t1, const SeqTable& t2, cudaStream_t s) {
  const int R = args.sh.R;
  if (R <= 32) return run<D, 32>(args, t1, t2, s);
  if (R <= 64) return run<D, 64>(args, t1, t2, s);
  if (R <= 128) return run<D, 128>(args, t1, t2, s);
  return run<D, 256>(args, t1, t2, s);
}

}  // namespace

kvsel_status launch_score_simt(const ScoreShape& sh, const SeqTable& t1, const SeqTable& t2, const void* q,
                               const void* k, float* scores, float* page_scores, float* lse, float2* part,
                               DeviceError* err, cudaStream_t s) {
  ScoreArgs args;
  args.sh = sh;
  args.q = static_cast<const __nv_bfloat16*>(q);
  args.k = static_cast<const __nv_bfloat16*>(k);
  args.scores = scores;
  args.page_scores = page_scores;
  args.lse = lse;
  args.part = part;
  args.err = err;
  if (t1.n_items <= 0 || t2.n_items <= 0) return KVSEL_ERR_INVALID_ARG;
  return sh.d == 64 ? run_d<64>(args, t1, t2, s) : run_d<128>(args, t1, t2, s);
}

kvsel_status launch_lse_combine(const ScoreShape& sh, const SeqTable& t1, float2* part, float* lse, cudaStream_t s) {
  ScoreArgs args{};
  args.sh = sh;
  args.part = part;
  args.lse = lse;
  const int64_t n_rows = (int64_t)t1.batch * sh.n_layers * sh.h_kv * sh.R;
  TraceScope ts("score_lse_combine", s);
  score_lse_combine<<<(unsigned)((n_rows + kThreads - 1) / kThreads), kThreads, 0, s>>>(args, t1, n_rows);
  return launch_status();
}

}  // namespace kvsel
