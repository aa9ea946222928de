// overlap.cu — cross-layer Top-k overlap counts for the anchor-selection DP
// (Kascade, euno.news summary, Methodology 4: the DP maximises the overlap of
// Top-k sets across layers on calibration data).
//
// Each (layer, unit) set becomes a bitmap of n_bits bits; one CTA per layer
// pair (i <= l) sums popc(bitmap_i & bitmap_l) over all units and words.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "kascade.h"

namespace kascade {
namespace {

__global__ void k_set_bits(const int32_t* __restrict__ sets, uint32_t* __restrict__ bm, int L,
                           int units, int topk, int n_bits, int words, unsigned int* err) {
  const size_t total = static_cast<size_t>(L) * units * topk;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t row = i / topk;   // (layer, unit)
    const int key = sets[i];
    if (key < 0 || key >= n_bits) {
      report_error(err, KASCADE_ERR_BAD_INPUT, 0x501);
      continue;
    }
    atomicOr(&bm[row * words + (key >> 5)], 1u << (key & 31));
  }
}

__global__ void k_pair_counts(const uint32_t* __restrict__ bm, long long* __restrict__ counts,
                              int L, int units, int words) {
  // blockIdx.x enumerates pairs i <= l in row-major upper-triangle order
  int p = blockIdx.x, i = 0;
  while (p >= L - i) {
    p -= L - i;
    ++i;
  }
  const int l = i + p;
  const size_t per_layer = static_cast<size_t>(units) * words;
  const uint32_t* a = bm + i * per_layer;
  const uint32_t* b = bm + l * per_layer;
  long long acc = 0;
  for (size_t w = threadIdx.x; w < per_layer; w += blockDim.x) acc += __popc(a[w] & b[w]);
  __shared__ long long red[32];
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long t = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += red[w];
    counts[static_cast<size_t>(i) * L + l] = t;
    counts[static_cast<size_t>(l) * L + i] = t;
  }
}

}  // namespace

cudaError_t launch_layer_overlap(const int32_t* sets, int L, int units, int topk, int n_bits,
                                 long long* counts, uint32_t* bitmaps, unsigned int* err,
                                 cudaStream_t st) {
  const int words = (n_bits + 31) / 32;
  const size_t bm_bytes = static_cast<size_t>(L) * units * words * 4;
  cudaError_t e = cudaMemsetAsync(bitmaps, 0, bm_bytes, st);
  if (e != cudaSuccess) return e;
  k_set_bits<<<152 * 8, 256, 0, st>>>(sets, bitmaps, L, units, topk, n_bits, words, err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_pair_counts<<<L * (L + 1) / 2, 512, 0, st>>>(bitmaps, counts, L, units, words);
  return cudaGetLastError();
}

}  // namespace kascade

extern "C" {

size_t kascade_overlap_workspace_size(int32_t n_layers, int32_t units, int32_t n_bits) {
  if (n_layers < 1 || units < 1 || n_bits < 1) return 0;
  const size_t words = (static_cast<size_t>(n_bits) + 31) / 32;
  return kascade::kWsStateBytes + static_cast<size_t>(n_layers) * units * words * 4;
}

kascade_status kascade_layer_overlap(const int32_t* sets, int32_t n_layers, int32_t units,
                                     int32_t topk, int32_t n_bits, int64_t* counts_out,
                                     void* ws, size_t ws_bytes, void* stream) {
  if (sets == nullptr || counts_out == nullptr || n_layers < 1 || units < 1 || topk < 1 ||
      n_bits < 1 || topk > n_bits)
    return KASCADE_ERR_INVALID_ARG;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) != 0 ||
      ws_bytes < kascade_overlap_workspace_size(n_layers, units, n_bits))
    return KASCADE_ERR_WORKSPACE;
  char* base = static_cast<char*>(ws);
  cudaError_t e = kascade::launch_layer_overlap(
      sets, n_layers, units, topk, n_bits, reinterpret_cast<long long*>(counts_out),
      reinterpret_cast<uint32_t*>(base + kascade::kWsStateBytes),
      reinterpret_cast<unsigned int*>(base), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KASCADE_OK : KASCADE_ERR_CUDA;
}

}  // extern "C"
