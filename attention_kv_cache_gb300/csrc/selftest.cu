// Self-test of the bounded device wait that every pipelined kernel of the library uses.
#include "internal.cuh"
#include "sm100.cuh"

namespace kvsel {
namespace {

// One CTA waits on an mbarrier with expected count 1.  Unless `arrive` is set, nothing arrives on it,
// so the wait must give up after `polls` polls and record KVSEL_ERR_TIMEOUT.
__global__ void selftest_wait_kernel(DeviceError* err, uint32_t polls, int arrive) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = sm100::smem_addr(&bar);
  if (threadIdx.x == 0) {
    sm100::mbar_init(b, 1);
    sm100::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 32 && arrive) sm100::mbar_arrive(b);
  if (threadIdx.x == 0 && !sm100::mbar_wait_n(b, 0, polls)) set_device_error(err, KVSEL_ERR_TIMEOUT, 0x5e1fu);
}

}  // namespace
}  // namespace kvsel

extern "C" KVSEL_API kvsel_status kvsel_selftest_bounded_wait(void* ws, uint32_t polls, int32_t arrive,
                                                              cudaStream_t stream) {
  if (ws == nullptr || ((uintptr_t)ws % KVSEL_WS_ALIGN) != 0) return KVSEL_ERR_WORKSPACE;
  if (polls == 0 || polls > (1u << 22)) return KVSEL_ERR_INVALID_ARG;
  kvsel::TraceScope ts("selftest_wait", stream);
  kvsel::selftest_wait_kernel<<<1, 64, 0, stream>>>(reinterpret_cast<kvsel::DeviceError*>(ws), polls, arrive != 0);
  return kvsel::launch_status();
}
