// kvsel_score_noalloc: kvsel_score with its scratch in a fixed array inside the library.
//
// Who needs this: callers that cannot allocate device memory themselves — a C
// plugin running inside a host program that owns every byte of the GPU's
// memory (a serving engine that has reserved HBM for its KV cache and hands
// out no extra buffers), or a latency-critical caller that must not pay
// cudaMalloc's implicit device-wide synchronisation on its hot path.  They
// pass inputs and outputs only; the row statistics and per-segment partials
// of the two scoring passes live in g_score_scratch below.
//
// The array is a file-scope __device__ variable, so every GPU that loads this
// library holds KVSEL_NOALLOC_SCRATCH_BYTES of it until the process exits.
// Its name in host code is only a host-side stand-in; the device address is
// looked up once per device with cudaGetSymbolAddress, with that device
// current, on the first call made while it is current.
#include <mutex>

#include "internal.cuh"

namespace {

constexpr size_t kScratchBytes = KVSEL_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % KVSEL_WS_ALIGN == 0, "scratch size must keep the workspace alignment");

static __device__ __align__(256) unsigned char g_score_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of g_score_scratch on the current device (looked up once per device).
kvsel_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVSEL_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KVSEL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_dev[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_score_scratch) != cudaSuccess || p == nullptr) return KVSEL_ERR_CUDA;
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return KVSEL_OK;
}

}  // namespace

extern "C" KVSEL_API kvsel_status kvsel_score_noalloc(const kvsel_desc* desc, const void* q, const void* k,
                                                      float* scores, float* page_scores,
                                                      cudaStream_t stream) {
  // Every argument check kvsel_score makes comes first, so a rejected call leaves nothing on the
  // stream and cannot clear the error word of an earlier call still in flight.
  kvsel_status st = kvsel::check_score_args(desc, q, k, scores, page_scores);
  if (st != KVSEL_OK) return st;
  size_t need = 0;
  if ((st = kvsel_workspace_size(desc, &need)) != KVSEL_OK) return st;
  if (need > kScratchBytes) return KVSEL_ERR_WORKSPACE;   // larger than the built-in scratch
  void* ws = nullptr;
  if ((st = scratch_on_current_device(&ws)) != KVSEL_OK) return st;
  // The array keeps the previous call's contents.  The scoring passes rewrite
  // every partial and row statistic before reading it; only the error word
  // must start at zero.
  if (cudaMemsetAsync(ws, 0, sizeof(kvsel::DeviceError), stream) != cudaSuccess) return KVSEL_ERR_CUDA;
  return kvsel_score(desc, q, k, scores, page_scores, ws, kScratchBytes, stream);
}

extern "C" KVSEL_API kvsel_status kvsel_noalloc_read_device_error(cudaStream_t stream) {
  void* ws = nullptr;
  kvsel_status st = scratch_on_current_device(&ws);
  if (st != KVSEL_OK) return st;
  return kvsel_read_device_error(ws, stream);
}
