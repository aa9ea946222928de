// shard.cu — sequence-sharded anchor decode: a shard's partials and their merge.
//
// The KV cache of every sequence is split along the key axis into contiguous
// shards in key order. A shard runs the anchor decode layer (exact attention
// and an exact per-head Top-k; Kascade, euno.news summary, Methodology 2) on
// its own keys; these kernels turn that into the shard's partials and merge
// the partials of all shards:
//   k_shard_finish : lse = log sum_j exp(s_j) of the shard (from the row's max
//                    and 1/sum of exp), and the local Top-k as global
//                    positions with their logits (gathered from the spill);
//   k_merge_out    : o = sum_s exp(lse_s - LSE) o_s, LSE = log sum_s exp(lse_s);
//   k_merge_scores : the shards' candidate logits of one row side by side, in
//                    shard order, for the ordinary Top-k kernel (positions in
//                    that row ascend with the global positions, so its
//                    lower-position tie rule is the global one); checks that
//                    the candidates ascend across shards;
//   k_merge_emit   : the selected row positions mapped back to global keys.
// The union of the shards' local Top-k sets holds the global Top-k (a key
// beaten by fewer than k keys overall is beaten by fewer than k keys of its
// shard), so the selection over the candidates is exact.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace kascade {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) k_shard_finish(const float* __restrict__ spill,
                                                           const float2* __restrict__ row_stat,
                                                           int n_s, int topk, int offset,
                                                           float* __restrict__ lse_out,
                                                           int32_t* __restrict__ cand_idx,
                                                           float* __restrict__ cand_scores) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  if (threadIdx.x == 0) {
    const float2 st = row_stat[r];   // (max, 1 / sum exp(s - max))
    lse_out[r] = st.x - logf(st.y);
  }
  const float* row = spill + static_cast<size_t>(r) * n_s;
  int32_t* ci = cand_idx + static_cast<size_t>(r) * topk;
  float* cs = cand_scores + static_cast<size_t>(r) * topk;
  for (int i = threadIdx.x; i < topk; i += kThreads) {
    const int local = ci[i];          // from the Top-k kernel: 0 <= local < n_s
    cs[i] = row[local];
    ci[i] = local + offset;
  }
}

template <typename T>
__device__ __forceinline__ float load_val(const T* p);
template <>
__device__ __forceinline__ float load_val<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_val<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void store_val(T* p, float x);
template <>
__device__ __forceinline__ void store_val<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void store_val<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

// One CTA per row (sequence, query head), one thread per output dimension.
template <typename T>
__global__ void k_merge_out(const T* __restrict__ outs, const float* __restrict__ lses,
                            int n_shards, int rows, int d, T* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, c = threadIdx.x;
  float m = -INFINITY;
  for (int s = 0; s < n_shards; ++s) m = fmaxf(m, lses[static_cast<size_t>(s) * rows + r]);
  float wsum = 0.f, acc = 0.f;
  for (int s = 0; s < n_shards; ++s) {
    const float w = expf(lses[static_cast<size_t>(s) * rows + r] - m);
    wsum += w;
    if (c < d) acc += w * load_val(outs + (static_cast<size_t>(s) * rows + r) * d + c);
  }
  if (c < d) store_val(out + static_cast<size_t>(r) * d + c, acc / wsum);
}

// scores [rows][S * topk] from cand_scores [S][rows][topk]; candidates must
// lie in [0, n_total) and ascend within and across shards.
__global__ void __launch_bounds__(kThreads) k_merge_scores(const int32_t* __restrict__ cand_idx,
                                                           const float* __restrict__ cand_scores,
                                                           int n_shards, int rows, int topk,
                                                           int n_total, float* __restrict__ scores,
                                                           unsigned int* err) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const int n = n_shards * topk;
  bool bad = false;
  for (int p = threadIdx.x; p < n; p += kThreads) {
    const int s = p / topk, i = p - s * topk;
    const size_t at = (static_cast<size_t>(s) * rows + r) * topk + i;
    scores[static_cast<size_t>(r) * n + p] = cand_scores[at];
    const int j = cand_idx[at];
    bad |= j < 0 || j >= n_total;
    if (p > 0) {
      const int sp = (p - 1) / topk, ip = (p - 1) - sp * topk;
      bad |= cand_idx[(static_cast<size_t>(sp) * rows + r) * topk + ip] >= j;
    }
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) report_error(err, KASCADE_ERR_BAD_INPUT, 0x601);
}

__global__ void __launch_bounds__(kThreads) k_merge_emit(const int32_t* __restrict__ pos,
                                                         const int32_t* __restrict__ cand_idx,
                                                         int rows, int topk,
                                                         int32_t* __restrict__ idx_out) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  for (int i = threadIdx.x; i < topk; i += kThreads) {
    const int p = pos[static_cast<size_t>(r) * topk + i];   // 0 <= p < S * topk
    const int s = p / topk, e = p - s * topk;
    idx_out[static_cast<size_t>(r) * topk + i] = cand_idx[(static_cast<size_t>(s) * rows + r) * topk + e];
  }
}

}  // namespace

cudaError_t launch_shard_finish(const float* spill, const float2* row_stat, int rows, int n_s,
                                int topk, int offset, float* lse_out, int32_t* cand_idx,
                                float* cand_scores, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  return launch_pdl(k_shard_finish, dim3(rows), dim3(kThreads), 0, st, spill, row_stat, n_s, topk,
                    offset, lse_out, cand_idx, cand_scores);
}

cudaError_t launch_merge_out(const void* outs, const float* lses, int n_shards, int rows, int d,
                             int dtype, void* out, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const dim3 block((d + 31) / 32 * 32);
  if (dtype == KASCADE_BF16)
    return launch_pdl(k_merge_out<__nv_bfloat16>, dim3(rows), block, 0, st,
                      static_cast<const __nv_bfloat16*>(outs), lses, n_shards, rows, d,
                      static_cast<__nv_bfloat16*>(out));
  return launch_pdl(k_merge_out<float>, dim3(rows), block, 0, st, static_cast<const float*>(outs),
                    lses, n_shards, rows, d, static_cast<float*>(out));
}

cudaError_t launch_merge_scores(const int32_t* cand_idx, const float* cand_scores, int n_shards,
                                int rows, int topk, int n_total, float* scores,
                                unsigned int* err, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  return launch_pdl(k_merge_scores, dim3(rows), dim3(kThreads), 0, st, cand_idx, cand_scores,
                    n_shards, rows, topk, n_total, scores, err);
}

cudaError_t launch_merge_emit(const int32_t* pos, const int32_t* cand_idx, int rows, int topk,
                              int32_t* idx_out, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  return launch_pdl(k_merge_emit, dim3(rows), dim3(kThreads), 0, st, pos, cand_idx, rows, topk,
                    idx_out);
}

}  // namespace kascade
