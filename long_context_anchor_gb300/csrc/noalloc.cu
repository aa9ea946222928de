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
// should therefore come before any stream capture. Every call shares the
// one array, and it keeps the last call's contents: each call clears the
// counters and the error word it needs (cudaMemsetAsync, no allocation), and
// calls that overlap on the GPU (concurrent streams) race on the array and
// must be serialised by the caller.
#include <cuda_runtime.h>
#include <math.h>
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
  if (desc == nullptr) return KASCADE_ERR_INVALID_ARG;
  const int B = desc->batch, Hq = desc->n_q_heads, Hkv = desc->n_kv_heads;
  const int d = desc->head_dim, N = desc->kv_len;
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || Hq % Hkv != 0 || Hq > kMaxQHeads)
    return KASCADE_ERR_INVALID_ARG;
  if (desc->dtype != KASCADE_BF16 || (d != 64 && d != 128)) return KASCADE_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KASCADE_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hkv * N >= (1ll << 31)) return KASCADE_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return KASCADE_ERR_INVALID_ARG;

  DecodeArgs a;
  memset(&a, 0, sizeof(a));
  int fill[kMaxQHeads] = {};
  for (int h = 0; h < Hq; ++h) {
    const int g = desc->group_map ? desc->group_map[h] : h / G;
    if (g < 0 || g >= Hkv || fill[g] >= G) return KASCADE_ERR_INVALID_ARG;
    a.heads[g * G + fill[g]++] = static_cast<int16_t>(h);
  }
  const int units = B * Hkv;
  a.chunk = decode_chunk_dense(units, N);
  a.S = (N + a.chunk - 1) / a.chunk;
  // Size check against the fixed scratch: header + counters, then partials.
  const size_t counters = static_cast<size_t>(units) * sizeof(unsigned int);
  const size_t partials = static_cast<size_t>(B) * Hq * a.S * (d + 4) * sizeof(float);
  if (sizeof(WsHeader) + counters > kCounterBytes ||
      kCounterBytes + partials > kNoAllocScratchBytes)
    return KASCADE_ERR_WORKSPACE;   // shape needs more than the 8 MiB scratch

  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return KASCADE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Counters and the error word must start at zero; partials are overwritten.
  if (cudaMemsetAsync(scratch, 0, sizeof(WsHeader) + counters, st) != cudaSuccess)
    return KASCADE_ERR_CUDA;
  char* base = static_cast<char*>(scratch);
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.err = reinterpret_cast<unsigned int*>(base);
  a.counters = reinterpret_cast<unsigned int*>(base + sizeof(WsHeader));
  a.part = reinterpret_cast<float*>(base + kCounterBytes);
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.N = N;
  a.G = G;
  a.topk = 1;
  a.scale = desc->scale > 0.f ? desc->scale : 1.0f / sqrtf(static_cast<float>(d));
  a.scale_log2 = a.scale * 1.4426950408889634f;
  return launch_decode_dense_bf16(a, d, false, st) == cudaSuccess ? KASCADE_OK : KASCADE_ERR_CUDA;
}
