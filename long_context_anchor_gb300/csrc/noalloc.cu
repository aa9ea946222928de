// noalloc.cu — dense decode attention for callers that cannot allocate.
//
// Every other entry point takes a caller-allocated workspace. Some callers
// cannot obtain one: code running where cudaMalloc is off limits (a custom
// allocator owns all device memory, or the call sits inside a host callback
// or a memory-pool section that forbids new allocations), or a plain C
// caller that only holds the tensors themselves. kascade_dense_decode_noalloc
// serves them: the split-K partials, the split counters and the device error
// word live in one file-scope device array of kNoAllocScratchBytes (8 MiB),
// which every GPU that loads the library holds until the process exits.
//
// The array's name is only a host-side stand-in in host code; its device
// address is fetched once per device with cudaGetSymbolAddress, on the first
// call made while that device is current, and cached. That first call
// should therefore come before any stream capture. The cache is keyed by the
// device ordinal, so the library must not be used across a cudaDeviceReset
// (the module, and with it the array, may be loaded at another address).
//
// Every call shares the one array, and it keeps the last call's contents:
// each call clears the split counters it needs (cudaMemsetAsync, no
// allocation), and calls that overlap on the GPU (concurrent streams) race on
// the array and must be serialised by the caller. The error word is not
// cleared by the calls: device faults accumulate there until
// kascade_noalloc_device_error reads and clears it.
#include <cuda_runtime.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "kascade.h"

namespace kascade {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
constexpr size_t kCounterBytes = 64 * 1024;   // header + split counters
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

inline bool aligned16(const void* p) {
  return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15) == 0;
}

}  // namespace
}  // namespace kascade

extern "C" kascade_status kascade_dense_decode_noalloc(const kascade_desc* desc, const void* q,
                                                       const void* k, const void* v, void* out,
                                                       void* stream) {
  using namespace kascade;
  Shape s;
  kascade_status r = check_desc(desc, s);   // the same limits as every other entry point
  if (r != KASCADE_OK) return r;
  if (s.dtype != KASCADE_BF16) return KASCADE_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return KASCADE_ERR_INVALID_ARG;

  DecodeArgs a;
  memset(&a, 0, sizeof(a));
  for (int i = 0; i < s.Hq; ++i) a.heads[i] = s.heads[i];
  const int units = s.B * s.Hkv;
  a.chunk = decode_chunk_dense(units, s.N);
  a.S = (s.N + a.chunk - 1) / a.chunk;
  // Size check against the fixed scratch: header + counters, then partials.
  const size_t counters = static_cast<size_t>(units) * sizeof(unsigned int);
  const size_t partials = static_cast<size_t>(s.B) * s.Hq * a.S * (s.d + 4) * sizeof(float);
  if (sizeof(WsHeader) + counters > kCounterBytes ||
      kCounterBytes + partials > kNoAllocScratchBytes)
    return KASCADE_ERR_WORKSPACE;   // shape needs more than the 8 MiB scratch

  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return KASCADE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(scratch);
  // The split counters must start at zero (a call cut short by a bounded wait
  // may have left some set); partials are overwritten; the error word stays.
  if (cudaMemsetAsync(base + sizeof(WsHeader), 0, counters, st) != cudaSuccess)
    return KASCADE_ERR_CUDA;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.err = reinterpret_cast<unsigned int*>(base);
  a.counters = reinterpret_cast<unsigned int*>(base + sizeof(WsHeader));
  a.part = reinterpret_cast<float*>(base + kCounterBytes);
  a.B = s.B;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.N = s.N;
  a.G = s.G;
  a.topk = 1;
  a.scale = s.scale;
  a.scale_log2 = s.scale * 1.4426950408889634f;
  return launch_decode_dense_bf16(a, s.d, false, st) == cudaSuccess ? KASCADE_OK
                                                                     : KASCADE_ERR_CUDA;
}

extern "C" kascade_status kascade_noalloc_device_error(void* stream) {
  using namespace kascade;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return KASCADE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return KASCADE_ERR_CUDA;
  unsigned int word[2] = {0u, 0u};
  // plain copies from and to the array: nothing is allocated
  if (cudaMemcpy(word, scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KASCADE_ERR_CUDA;
  if (word[0] != 0) {
    const unsigned int zero[2] = {0u, 0u};
    if (cudaMemcpy(scratch, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return KASCADE_ERR_CUDA;
  }
  if (word[0] & (1u << KASCADE_ERR_TIMEOUT)) return KASCADE_ERR_TIMEOUT;
  if (word[0] & (1u << KASCADE_ERR_BAD_INPUT)) return KASCADE_ERR_BAD_INPUT;
  return KASCADE_OK;
}
