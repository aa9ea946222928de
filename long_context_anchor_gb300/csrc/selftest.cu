// selftest.cu — the failure path of the bounded waits, for tests.
//
// Every kernel of the library waits on mbarriers through mbar_wait, which
// gives up after a bounded time, records KASCADE_ERR_TIMEOUT in the
// workspace's error word and lets the kernel return, so a lost arrival never
// hangs the GPU. This entry point runs that wait on a barrier nothing arrives
// on, so a test can see the timeout reported and the context still usable.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "kascade.h"

namespace kascade {
namespace {

__global__ void k_wait_timeout(unsigned int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, err, 0x901);   // phase 0 never completes
}

}  // namespace
}  // namespace kascade

extern "C" kascade_status kascade_check_wait_timeout(void* ws, size_t ws_bytes, void* stream) {
  using namespace kascade;
  if (ws == nullptr || ws_bytes < sizeof(WsHeader)) return KASCADE_ERR_WORKSPACE;
  unsigned int* err = static_cast<unsigned int*>(ws);
  k_wait_timeout<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err);
  return cudaGetLastError() == cudaSuccess ? KASCADE_OK : KASCADE_ERR_CUDA;
}
