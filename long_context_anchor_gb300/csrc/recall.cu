// recall.cu — attention-mass-recall similarity for the anchor DP.
//
// The pages choose anchors by a DP that maximises the "overlap (similarity)
// of top-k sets across layers" (euno.news summary, Methodology 4) without
// giving a formula. Besides the set overlap (overlap.cu) the library offers
// the mass of layer l's exact attention that layer i's set keeps:
//   M[i][l] = mean over (sequence, query head) of sum_{j in S_i} p_l[j],
// with p_l the softmax of layer l's scaled logits over all N keys. Layer l's
// logits are in the anchor's spill right after its anchor call, so the DP
// entries M[i][l], i <= l, are summed then, against the sets of layers 0..l.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace kascade {
namespace {

constexpr float kLog2eR = 1.4426950408889634f;

struct KvTable {
  int16_t head_kv[kMaxQHeads];   // KV head of each query head
};

// Block (r, i): row r = b*Hq + h of layer l's logits; the set of layer i for
// that head (its own, or its KV head's when pooled). part[(l*L + i)*rows + r]
// = sum over the set of exp(s - m) / sum_row exp(s - m).
__global__ void __launch_bounds__(256) k_mass_recall(const float* __restrict__ s,
                                                     const float2* __restrict__ row_stat,
                                                     const int32_t* __restrict__ sets,
                                                     size_t per_layer, int topk, int n, int Hq,
                                                     int Hkv, int pooled, int layer, int n_layers,
                                                     const __grid_constant__ KvTable kv,
                                                     float* __restrict__ part,
                                                     unsigned int* err) {
  __shared__ float red[8];
  const int r = blockIdx.x, i = blockIdx.y, rows = gridDim.x;
  const int b = r / Hq, h = r % Hq;
  const int set_row = pooled ? b * Hkv + kv.head_kv[h] : r;
  const int32_t* set = sets + static_cast<size_t>(i) * per_layer + static_cast<size_t>(set_row) * topk;
  const float* row = s + static_cast<size_t>(r) * n;
  const float2 st = row_stat[r];
  float acc = 0.f;
  for (int e = threadIdx.x; e < topk; e += blockDim.x) {
    const int j = __ldg(set + e);
    if (j < 0 || j >= n) {
      report_error(err, KASCADE_ERR_BAD_INPUT, 0x801);
      continue;
    }
    acc += exp2f((__ldg(row + j) - st.x) * kLog2eR) * st.y;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) tot += red[w];
    part[(static_cast<size_t>(layer) * n_layers + i) * rows + r] = tot;
  }
}

// sim[i*L + l] = mean over rows of part[(l*L + i)*rows + r] for i <= l (in
// float64, rows in order), 0 for i > l.
__global__ void __launch_bounds__(256) k_recall_reduce(const float* __restrict__ part, int n_layers,
                                                       int rows, double* __restrict__ sim) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n_layers * n_layers) return;
  const int i = e / n_layers, l = e % n_layers;
  double tot = 0.0;
  if (i <= l) {
    const float* p = part + (static_cast<size_t>(l) * n_layers + i) * rows;
    for (int r = 0; r < rows; ++r) tot += static_cast<double>(p[r]);
    tot /= rows;
  }
  sim[e] = tot;
}

}  // namespace

cudaError_t launch_mass_recall(const float* spill, const float2* row_stat, const int32_t* sets,
                               size_t per_layer, int topk, int B, int Hq, int Hkv, int N,
                               int pooled, const int16_t* head_kv, int layer, int n_layers,
                               float* part, unsigned int* err, cudaStream_t st) {
  if (B < 1 || Hq < 1 || Hq > kMaxQHeads || topk < 1 || layer < 0 || layer >= n_layers)
    return cudaErrorInvalidValue;
  KvTable kv{};
  for (int h = 0; h < Hq; ++h) kv.head_kv[h] = head_kv[h];
  k_mass_recall<<<dim3(B * Hq, layer + 1), 256, 0, st>>>(spill, row_stat, sets, per_layer, topk, N,
                                                         Hq, Hkv, pooled, layer, n_layers, kv,
                                                         part, err);
  return cudaGetLastError();
}

cudaError_t launch_recall_reduce(const float* part, int n_layers, int rows, double* sim,
                                 cudaStream_t st) {
  const int n = n_layers * n_layers;
  k_recall_reduce<<<(n + 255) / 256, 256, 0, st>>>(part, n_layers, rows, sim);
  return cudaGetLastError();
}

}  // namespace kascade
