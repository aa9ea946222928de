// pool.cu — scores of GQA-pooled index sets (one set per KV head).
//
// The Kascade pages give every attention head its own Top-k list (euno.news
// summary, Methodology 5) and run GQA models. In pooled mode the query heads
// of one KV head share a list, ranked by the sum of their post-softmax
// weights: decode w[b,g,j] = sum_{h: g(h)=g} softmax_j(s[b,h,:]), prefill the
// sum of the group's tile weights w_{t,h,j}. Both kernels here are plain
// HBM/L2 streams over fp32 rows the anchor layer has just written.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace kascade {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
#define kNegInf (__int_as_float(0xff800000u))

struct HeadTable {
  int16_t heads[kMaxQHeads];   // heads[g*G + slot]
};

// (max, sum of exp(x - max)) pairs, merged exactly as the online softmax does.
__device__ __forceinline__ void stat_merge(float& m, float& s, float m2, float s2) {
  if (m2 == kNegInf) return;
  if (m == kNegInf) {
    m = m2;
    s = s2;
    return;
  }
  const float mx = fmaxf(m, m2);
  s = s * exp2f((m - mx) * kLog2e) + s2 * exp2f((m2 - mx) * kLog2e);
  m = mx;
}

// One CTA per logit row: row_stat[r] = (max_j s_rj, 1 / sum_j exp(s_rj - max)).
// Each thread takes kStatUnroll keys per step with independent loads (the row
// was just written and mostly sits in L2, so the loop is load-latency bound
// unless several loads are in flight), then folds them into its running
// (max, sum). A NaN logit makes the sum NaN, so every pooled weight of its
// group is NaN and the Top-k that follows reports it.
constexpr int kStatThreads = 512, kStatUnroll = 8;
__global__ void __launch_bounds__(kStatThreads) k_row_stat(const float* __restrict__ s, int n,
                                                           float2* __restrict__ row_stat) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sm[kStatThreads / 32], ss[kStatThreads / 32];
  const float* row = s + static_cast<size_t>(blockIdx.x) * n;
  float m = kNegInf, sum = 0.f;
  for (int j0 = threadIdx.x; j0 < n; j0 += kStatThreads * kStatUnroll) {
    float x[kStatUnroll];
#pragma unroll
    for (int u = 0; u < kStatUnroll; ++u) {
      const int j = j0 + u * kStatThreads;
      x[u] = j < n ? __ldg(row + j) : kNegInf;
    }
    float lm = x[0];
#pragma unroll
    for (int u = 1; u < kStatUnroll; ++u) lm = fmaxf(lm, x[u]);
    if (lm > m) {
      sum = (m == kNegInf) ? 0.f : sum * exp2f((m - lm) * kLog2e);
      m = lm;
    }
    if (m != kNegInf) {
#pragma unroll
      for (int u = 0; u < kStatUnroll; ++u) sum += exp2f((x[u] - m) * kLog2e);
    } else {
#pragma unroll
      for (int u = 0; u < kStatUnroll; ++u)
        if (x[u] != kNegInf) sum += exp2f(x[u]);   // NaN reaches the sum
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, sum, off);
    stat_merge(m, sum, m2, s2);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sm[warp] = m;
    ss[warp] = sum;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = sm[0], S = ss[0];
    for (int w = 1; w < kStatThreads / 32; ++w) stat_merge(M, S, sm[w], ss[w]);
    row_stat[blockIdx.x] = make_float2(M, 1.f / S);
  }
}

// w[u, j] = sum over the group's slots of exp(s[row, j] - max_row) / sum_row,
// u = b*Hkv + g, row = b*Hq + heads[g*G + slot]. Block (x, u) covers keys
// [1024 x, 1024 x + 1024), four per thread, coalesced.
__global__ void __launch_bounds__(256) k_pool_decode(const float* __restrict__ s,
                                                     const float2* __restrict__ row_stat,
                                                     float* __restrict__ w,
                                                     const __grid_constant__ HeadTable ht,
                                                     int Hq, int Hkv, int G, int n) {
  pdl_wait();
  pdl_trigger();
  const int u = blockIdx.y, b = u / Hkv, g = u % Hkv;
  const int j0 = blockIdx.x * 1024 + threadIdx.x;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int slot = 0; slot < G; ++slot) {
    const int r = b * Hq + ht.heads[g * G + slot];
    const float2 st = row_stat[r];
    const float* row = s + static_cast<size_t>(r) * n;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = j0 + 256 * i;
      if (j < n) acc[i] += exp2f((__ldg(row + j) - st.x) * kLog2e) * st.y;
    }
  }
  float* out = w + static_cast<size_t>(u) * n;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = j0 + 256 * i;
    if (j < n) out[j] = acc[i];
  }
}

// w_pool[u][e] = sum over the group's slots of w[b*Hq + heads[g*G + slot]][e].
__global__ void __launch_bounds__(256) k_pool_prefill(const float* __restrict__ w,
                                                      float* __restrict__ w_pool,
                                                      const __grid_constant__ HeadTable ht,
                                                      int Hq, int Hkv, int G, size_t per_bh) {
  const int u = blockIdx.y, b = u / Hkv, g = u % Hkv;
  const size_t e0 = static_cast<size_t>(blockIdx.x) * 1024 + threadIdx.x;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int slot = 0; slot < G; ++slot) {
    const float* row =
        w + static_cast<size_t>(b * Hq + ht.heads[g * G + slot]) * per_bh;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const size_t e = e0 + 256 * i;
      if (e < per_bh) acc[i] += __ldg(row + e);
    }
  }
  float* out = w_pool + static_cast<size_t>(u) * per_bh;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const size_t e = e0 + 256 * i;
    if (e < per_bh) out[e] = acc[i];
  }
}

HeadTable make_table(const int16_t* heads, int Hq) {
  HeadTable t{};
  for (int i = 0; i < Hq && i < kMaxQHeads; ++i) t.heads[i] = heads[i];
  return t;
}

}  // namespace

cudaError_t launch_pool_decode(const float* spill, float2* row_stat, float* w, bool stats_given,
                               const int16_t* heads, int B, int Hq, int Hkv, int G, int N,
                               cudaStream_t st) {
  if (B < 1 || Hq < 1 || Hkv < 1 || G < 1 || N < 1 || Hq != Hkv * G || Hq > kMaxQHeads)
    return cudaErrorInvalidValue;
  const HeadTable ht = make_table(heads, Hq);
  if (!stats_given) {
    const cudaError_t e = launch_pdl(k_row_stat, dim3(B * Hq), dim3(kStatThreads), 0, st, spill,
                                     N, row_stat);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(k_pool_decode, dim3((N + 1023) / 1024, B * Hkv), dim3(256), 0, st, spill,
                    static_cast<const float2*>(row_stat), w, ht, Hq, Hkv, G, N);
}

cudaError_t launch_row_stat(const float* s, int rows, int n, float2* row_stat, cudaStream_t st) {
  if (rows < 1 || n < 1) return cudaErrorInvalidValue;
  k_row_stat<<<rows, kStatThreads, 0, st>>>(s, n, row_stat);
  return cudaGetLastError();
}

cudaError_t launch_pool_prefill(const float* w, float* w_pool, const int16_t* heads, int B,
                                int Hq, int Hkv, int G, size_t per_bh, cudaStream_t st) {
  if (B < 1 || Hq < 1 || Hkv < 1 || G < 1 || Hq != Hkv * G || Hq > kMaxQHeads || per_bh == 0)
    return cudaErrorInvalidValue;
  const size_t blocks = (per_bh + 1023) / 1024;
  if (blocks > 0x7fffffffu) return cudaErrorInvalidValue;
  const HeadTable ht = make_table(heads, Hq);
  k_pool_prefill<<<dim3(static_cast<unsigned int>(blocks), B * Hkv), 256, 0, st>>>(
      w, w_pool, ht, Hq, Hkv, G, per_bh);
  return cudaGetLastError();
}

}  // namespace kascade
