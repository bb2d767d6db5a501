/*
 * A plain C caller of libkvsel: score -> top-k -> compact through the C ABI alone (no torch, no
 * Python), on a small problem with a planted key, checking what the method fixes without an
 * oracle:
 *   - each window row's softmax sums to 1, so a group's column mass over the prefix lies in
 *     (0, G * W] and every score is >= 0;
 *   - a key aligned with every window query of a group ranks first in that group;
 *   - the kept prefix positions are ascending, in range, hold the planted key, and score at least
 *     as high as every position not kept; the window positions L .. L + W - 1 follow them;
 *   - the compacted K and V rows are the source rows, bit for bit, whether V is read from device
 *     memory or from pinned host memory.
 * Built and run by tests/test_c_client.py; prints "c client ok" and exits 0 when every check holds.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "kvsel.h"

#define KV_CHECK(x)                                                                          \
  do {                                                                                       \
    kvsel_status s_ = (x);                                                                   \
    if (s_ != KVSEL_OK) {                                                                    \
      fprintf(stderr, "%s:%d %s -> %s\n", __FILE__, __LINE__, #x, kvsel_status_string(s_)); \
      return 1;                                                                              \
    }                                                                                        \
  } while (0)
#define CUDA_CHECK(x)                                                                     \
  do {                                                                                    \
    cudaError_t e_ = (x);                                                                 \
    if (e_ != cudaSuccess) {                                                              \
      fprintf(stderr, "%s:%d %s -> %s\n", __FILE__, __LINE__, #x, cudaGetErrorString(e_)); \
      return 1;                                                                           \
    }                                                                                     \
  } while (0)
#define EXPECT(c)                                                           \
  do {                                                                      \
    if (!(c)) {                                                             \
      fprintf(stderr, "%s:%d check failed: %s\n", __FILE__, __LINE__, #c); \
      return 1;                                                             \
    }                                                                       \
  } while (0)

/* float -> bfloat16 bits, round to nearest even (finite inputs only) */
static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static uint32_t rng_state = 0x6B767365u;
static float uniform_pm1(void) { /* xorshift32, uniform in [-1, 1) */
  rng_state ^= rng_state << 13;
  rng_state ^= rng_state >> 17;
  rng_state ^= rng_state << 5;
  return (float)(rng_state >> 8) * (2.0f / 16777216.0f) - 1.0f;
}

int main(void) {
  enum { LAYERS = 2, HQ = 8, HKV = 2, D = 128, W = 16, KEEP = 32 };
  const int G = HQ / HKV;
  const int64_t L = 1000, N = 1000 + W;
  const int64_t PLANT = 377;
  const int N_SEL = KEEP + W;

  kvsel_desc desc;
  memset(&desc, 0, sizeof desc);
  desc.n_layers = LAYERS;
  desc.h_q = HQ;
  desc.h_kv = HKV;
  desc.head_dim = D;
  desc.window = W;
  desc.batch = 1;
  desc.prefix_lens = &L;
  desc.group_reduce = KVSEL_REDUCE_SUM;
  desc.pool_k = 1;
  desc.page_size = 1;
  desc.page_reduce = KVSEL_REDUCE_MAX;
  desc.pool_type = KVSEL_POOL_MAX;
  desc.score_mode = KVSEL_SCORE_SOFTMAX;

  /* q [1][LAYERS][HQ][W][D]; k, v [LAYERS][HKV][N][D]: queries share a direction u (unit, spread
   * over every channel) plus small noise; keys are noise; key PLANT of every (layer, group) is 20 u */
  const size_t nq = (size_t)LAYERS * HQ * W * D, nk = (size_t)LAYERS * HKV * N * D;
  uint16_t* q = malloc(nq * 2);
  uint16_t* k = malloc(nk * 2);
  uint16_t* v = malloc(nk * 2);
  EXPECT(q && k && v);
  const float u = 1.0f / sqrtf((float)D);
  for (size_t i = 0; i < nq; ++i) q[i] = to_bf16(u + 0.05f * uniform_pm1());
  for (size_t i = 0; i < nk; ++i) {
    k[i] = to_bf16(0.5f * uniform_pm1());
    v[i] = to_bf16(uniform_pm1());
  }
  for (int l = 0; l < LAYERS; ++l)
    for (int g = 0; g < HKV; ++g)
      for (int c = 0; c < D; ++c) k[(((size_t)l * HKV + g) * N + PLANT) * D + c] = to_bf16(20.0f * u);

  void *dq, *dk, *dv, *dws, *dko, *dvo;
  float* dscores;
  int32_t* didx;
  size_t ws_bytes = 0;
  KV_CHECK(kvsel_workspace_size(&desc, &ws_bytes));
  const size_t n_scores = (size_t)LAYERS * HKV * L, n_idx = (size_t)LAYERS * HKV * N_SEL;
  const size_t n_out = n_idx * D;
  CUDA_CHECK(cudaMalloc(&dq, nq * 2));
  CUDA_CHECK(cudaMalloc(&dk, nk * 2));
  CUDA_CHECK(cudaMalloc(&dv, nk * 2));
  CUDA_CHECK(cudaMalloc(&dws, ws_bytes));   /* cudaMalloc's alignment covers KVSEL_WS_ALIGN */
  CUDA_CHECK(cudaMalloc((void**)&dscores, n_scores * 4));
  CUDA_CHECK(cudaMalloc((void**)&didx, n_idx * 4));
  CUDA_CHECK(cudaMalloc(&dko, n_out * 2));
  CUDA_CHECK(cudaMalloc(&dvo, n_out * 2));
  CUDA_CHECK(cudaMemset(dws, 0, ws_bytes));
  CUDA_CHECK(cudaMemcpy(dq, q, nq * 2, cudaMemcpyHostToDevice));
  CUDA_CHECK(cudaMemcpy(dk, k, nk * 2, cudaMemcpyHostToDevice));
  CUDA_CHECK(cudaMemcpy(dv, v, nk * 2, cudaMemcpyHostToDevice));

  KV_CHECK(kvsel_score(&desc, dq, dk, dscores, NULL, dws, ws_bytes, 0));
  KV_CHECK(kvsel_topk(&desc, dscores, LAYERS, KEEP, 0, didx, dws, ws_bytes, 0));
  KV_CHECK(kvsel_compact(&desc, dk, dv, didx, LAYERS, N_SEL, dko, dvo, dws, 0));
  KV_CHECK(kvsel_read_device_error(dws, 0));

  float* scores = malloc(n_scores * 4);
  int32_t* idx = malloc(n_idx * 4);
  uint16_t* ko = malloc(n_out * 2);
  uint16_t* vo = malloc(n_out * 2);
  EXPECT(scores && idx && ko && vo);
  CUDA_CHECK(cudaMemcpy(scores, dscores, n_scores * 4, cudaMemcpyDeviceToHost));
  CUDA_CHECK(cudaMemcpy(idx, didx, n_idx * 4, cudaMemcpyDeviceToHost));
  CUDA_CHECK(cudaMemcpy(ko, dko, n_out * 2, cudaMemcpyDeviceToHost));
  CUDA_CHECK(cudaMemcpy(vo, dvo, n_out * 2, cudaMemcpyDeviceToHost));

  for (int l = 0; l < LAYERS; ++l) {
    for (int g = 0; g < HKV; ++g) {
      const float* s = scores + ((size_t)l * HKV + g) * L;
      const int32_t* sel = idx + ((size_t)l * HKV + g) * N_SEL;
      double mass = 0.0;
      int64_t best = 0;
      for (int64_t t = 0; t < L; ++t) {
        EXPECT(s[t] >= 0.0f);
        mass += s[t];
        if (s[t] > s[best]) best = t;
      }
      EXPECT(mass > 0.0 && mass <= (double)G * W * (1.0 + 1e-3));
      EXPECT(best == PLANT);
      char* kept = calloc((size_t)L, 1);
      EXPECT(kept);
      int has_plant = 0;
      float min_kept = INFINITY;
      for (int i = 0; i < KEEP; ++i) {
        EXPECT(sel[i] >= 0 && sel[i] < L);
        if (i > 0) EXPECT(sel[i] > sel[i - 1]);
        kept[sel[i]] = 1;
        has_plant |= sel[i] == PLANT;
        if (s[sel[i]] < min_kept) min_kept = s[sel[i]];
      }
      EXPECT(has_plant);
      for (int64_t t = 0; t < L; ++t)
        if (!kept[t]) EXPECT(s[t] <= min_kept);
      free(kept);
      for (int j = 0; j < W; ++j) EXPECT(sel[KEEP + j] == L + j);
      for (int i = 0; i < N_SEL; ++i) {
        const size_t src = (((size_t)l * HKV + g) * N + sel[i]) * D;
        const size_t dst = (((size_t)l * HKV + g) * N_SEL + i) * D;
        EXPECT(memcmp(ko + dst, k + src, D * 2) == 0);
        EXPECT(memcmp(vo + dst, v + src, D * 2) == 0);
      }
    }
  }

  /* V in pinned host memory: the gather reads the kept rows over the host link */
  void* vh = NULL;
  CUDA_CHECK(cudaHostAlloc(&vh, nk * 2, cudaHostAllocDefault));
  memcpy(vh, v, nk * 2);
  CUDA_CHECK(cudaMemset(dvo, 0, n_out * 2));
  KV_CHECK(kvsel_compact(&desc, dk, vh, didx, LAYERS, N_SEL, dko, dvo, dws, 0));
  KV_CHECK(kvsel_read_device_error(dws, 0));
  uint16_t* vo2 = malloc(n_out * 2);
  EXPECT(vo2);
  CUDA_CHECK(cudaMemcpy(vo2, dvo, n_out * 2, cudaMemcpyDeviceToHost));
  EXPECT(memcmp(vo2, vo, n_out * 2) == 0);
  /* pageable host memory is refused before any launch */
  const int64_t launches = kvsel_launch_count();
  EXPECT(kvsel_compact(&desc, dk, v, didx, LAYERS, N_SEL, dko, dvo, dws, 0) == KVSEL_ERR_INVALID_ARG);
  EXPECT(kvsel_launch_count() == launches);

  cudaFreeHost(vh);
  cudaFree(dq);
  cudaFree(dk);
  cudaFree(dv);
  cudaFree(dws);
  cudaFree(dscores);
  cudaFree(didx);
  cudaFree(dko);
  cudaFree(dvo);
  free(q);
  free(k);
  free(v);
  free(scores);
  free(idx);
  free(ko);
  free(vo);
  free(vo2);
  printf("c client ok (%s)\n", kvsel_version());
  return 0;
}
