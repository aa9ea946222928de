// topk.cu — exact Top-k of fp32 rows (Kascade anchor layers take an exact,
// head-aware Top-k; euno.news summary, Key Contributions and Methodology 2,
// 5). Rule: larger score first, lower index wins a tie, -0 == +0; output
// ascending positions.
//
// One CTA (32 warps) per row:
//   1. scores become order-preserving uint32 keys; rows up to 32768 entries
//      are staged in shared memory once, longer rows are re-read (from L2);
//   2. radix select on 11/11/10-bit digits with warp-aggregated shared
//      histograms; as soon as the bin holding the k-th key fits, its members
//      are compacted into a shared candidate list and the remaining digits
//      run on the candidates only;
//   3. with the k-th key T known, the row is split into 32 warp segments;
//      per-segment counts of keys > T and == T are scanned, and each warp
//      writes its selected positions in index order using ballots, taking
//      keys == T in index order until k are selected.
// Prefill rows are the packed tile weights of one (sequence, head, tile):
// length L_t = min(N, 128(t+1)), k_t = min(k, L_t), -1 padding after k_t.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace kascade {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kRowCap = 32768;   // entries staged in shared memory
constexpr int kCandCap = 8192;   // candidate (key, position) pairs

struct RowDesc {
  const float* ptr;
  int len;
  int k;
};

__device__ __forceinline__ RowDesc row_desc(const TopkArgs& a, int r) {
  RowDesc d;
  if (a.prefill_tiles == 0) {
    d.ptr = a.scores + static_cast<size_t>(r) * a.n;
    d.len = a.n;
  } else {
    // packed rows of one (sequence, head): tile t starts at (tile/2)*t*(t+1)
    const int nT = a.prefill_tiles;
    const int bh = r / nT, t = r % nT;
    const size_t per_bh = static_cast<size_t>(a.tile / 2) * (nT - 1) * nT + a.n;
    d.ptr = a.scores + bh * per_bh + static_cast<size_t>(a.tile / 2) * t * (t + 1);
    d.len = min(a.n, a.tile * (t + 1));
  }
  d.k = min(a.k, d.len);
  return d;
}

// Inclusive block scan of one int per thread.
__device__ __forceinline__ int block_incl_scan(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += o;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  const int base = warp > 0 ? warp_tot[warp - 1] : 0;
  __syncthreads();
  return v + base;
}

__device__ __forceinline__ void hist_add(uint32_t* hist, bool active, uint32_t bin) {
  const unsigned int mask = __ballot_sync(0xffffffffu, active);
  if (active) {
    const unsigned int peers = __match_any_sync(mask, bin);
    if (static_cast<int>(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
  }
}

__global__ void __launch_bounds__(kThreads, 1) k_topk(const __grid_constant__ TopkArgs a) {
  extern __shared__ uint32_t sm[];
  uint32_t* hist = sm;                                                     // [2048]
  uint32_t* cand_key = hist + 2048;                                        // [kCandCap]
  int32_t* cand_pos = reinterpret_cast<int32_t*>(cand_key + kCandCap);     // [kCandCap]
  uint32_t* row_keys = reinterpret_cast<uint32_t*>(cand_pos + kCandCap);   // [len] if staged
  __shared__ int warp_tot[32];
  __shared__ int seg_gt[kWarps], seg_eq[kWarps];
  __shared__ int s_ncand, s_bin, s_above;

  const int r = blockIdx.x;
  const RowDesc rd = row_desc(a, r);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* out = a.idx_out + static_cast<size_t>(r) * a.k_stride;

  if (rd.k >= rd.len) {   // the whole prefix is selected
    for (int j = tid; j < a.k_stride; j += kThreads) out[j] = (j < rd.len) ? j : -1;
    return;
  }
  const bool staged = a.n <= kRowCap;   // shared memory is sized for a.n >= rd.len
  if (tid == 0) s_ncand = 0;
  if (staged) {
    bool bad = false;
    for (int j = tid; j < rd.len; j += kThreads) {
      const float f = __ldg(rd.ptr + j);
      bad |= isnan(f);
      row_keys[j] = float_key(f);
    }
    if (__syncthreads_or(bad) && tid == 0) report_error(a.err, KASCADE_ERR_BAD_INPUT, 0x401);
  } else {
    __syncthreads();
  }
  auto key_at = [&](int j) -> uint32_t {
    return staged ? row_keys[j] : float_key(__ldg(rd.ptr + j));
  };

  uint32_t prefix = 0, pmask = 0;
  int c_gt = 0;
  bool in_cands = false;
  const int seg = (((rd.len + kWarps - 1) / kWarps) + 31) & ~31;
  const int seg0 = warp * seg, seg1 = min(rd.len, seg0 + seg);

  for (int d = 0; d < 3; ++d) {
    const int nb = d < 2 ? 2048 : 1024;
    const int sh = d == 0 ? 21 : (d == 1 ? 10 : 0);
    for (int i = tid; i < nb; i += kThreads) hist[i] = 0u;
    __syncthreads();
    if (in_cands) {
      const int nc = s_ncand;
      for (int i = tid; i < nc; i += kThreads) {
        const uint32_t key = cand_key[i];
        if ((key & pmask) == prefix) atomicAdd(&hist[(key >> sh) & (nb - 1)], 1u);
      }
    } else {
      bool bad = false;
      for (int j0 = 0; j0 < rd.len; j0 += kThreads) {
        const int j = j0 + tid;
        uint32_t key = 0;
        bool act = false;
        if (j < rd.len) {
          if (!staged && d == 0) {
            const float f = __ldg(rd.ptr + j);
            bad |= isnan(f);
            key = float_key(f);
          } else {
            key = key_at(j);
          }
          act = (key & pmask) == prefix;
        }
        hist_add(hist, act, (key >> sh) & (nb - 1));
      }
      if (bad) report_error(a.err, KASCADE_ERR_BAD_INPUT, 0x402);
    }
    __syncthreads();
    // Locate the bin holding rank `need` counting from the top bin down.
    const int need = rd.k - c_gt;
    const int b_hi = nb - 1 - 2 * tid;   // this thread owns bins b_hi, b_hi-1
    int h0 = 0, h1 = 0;
    if (b_hi >= 0) h0 = static_cast<int>(hist[b_hi]);
    if (b_hi - 1 >= 0) h1 = static_cast<int>(hist[b_hi - 1]);
    const int incl = block_incl_scan(h0 + h1, warp_tot);
    const int excl = incl - h0 - h1;
    if (b_hi >= 0) {
      if (excl < need && need <= excl + h0) {
        s_bin = b_hi;
        s_above = excl;
      } else if (b_hi - 1 >= 0 && excl + h0 < need && need <= excl + h0 + h1) {
        s_bin = b_hi - 1;
        s_above = excl + h0;
      }
    }
    __syncthreads();
    const int bin = s_bin;
    c_gt += s_above;
    prefix |= static_cast<uint32_t>(bin) << sh;
    pmask |= static_cast<uint32_t>(nb - 1) << sh;
    const int cnt_bin = static_cast<int>(hist[bin]);
    __syncthreads();
    if (!in_cands && d < 2 && cnt_bin <= kCandCap) {
      // Compact the bin's members; count keys above the prefix per segment.
      int above = 0;
      for (int j0 = seg0; j0 < seg0 + seg; j0 += 32) {
        const int j = j0 + lane;
        uint32_t key = 0;
        bool is_c = false;
        if (j < seg1) {
          key = key_at(j);
          const uint32_t hi = key & pmask;
          above += hi > prefix;
          is_c = hi == prefix;
        }
        const unsigned int bal = __ballot_sync(0xffffffffu, is_c);
        int base = 0;
        if (lane == 0 && bal) base = atomicAdd(&s_ncand, __popc(bal));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (is_c) {
          const int p = base + __popc(bal & ((1u << lane) - 1u));
          cand_key[p] = key;
          cand_pos[p] = j;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) above += __shfl_xor_sync(0xffffffffu, above, off);
      if (lane == 0) seg_gt[warp] = above;
      in_cands = true;
      __syncthreads();
    }
  }
  const uint32_t T = prefix;   // the k-th largest key
  // Per-segment counts of keys > T and == T.
  if (in_cands) {
    if (tid < kWarps) seg_eq[tid] = 0;
    __syncthreads();
    const int nc = s_ncand;
    for (int i = tid; i < nc; i += kThreads) {
      const uint32_t key = cand_key[i];
      const int sgi = cand_pos[i] / seg;
      if (key > T) atomicAdd(&seg_gt[sgi], 1);
      else if (key == T) atomicAdd(&seg_eq[sgi], 1);
    }
  } else {
    int gt = 0, eq = 0;
    for (int j = seg0 + lane; j < seg1; j += 32) {
      const uint32_t key = key_at(j);
      gt += key > T;
      eq += key == T;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      gt += __shfl_xor_sync(0xffffffffu, gt, off);
      eq += __shfl_xor_sync(0xffffffffu, eq, off);
    }
    if (lane == 0) {
      seg_gt[warp] = gt;
      seg_eq[warp] = eq;
    }
  }
  __syncthreads();
  int gt_before = 0, eq_before = 0, gt_total = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) {
      gt_before += seg_gt[w];
      eq_before += seg_eq[w];
    }
    gt_total += seg_gt[w];
  }
  const int need_eq = rd.k - gt_total;
  // Ordered write of the selected positions.
  int run_gt = 0, run_eq = 0;
  for (int j0 = seg0; j0 < seg0 + seg; j0 += 32) {
    const int j = j0 + lane;
    bool gt = false, eq = false;
    if (j < seg1) {
      const uint32_t key = key_at(j);
      gt = key > T;
      eq = key == T;
    }
    const unsigned int bg = __ballot_sync(0xffffffffu, gt);
    const unsigned int be = __ballot_sync(0xffffffffu, eq);
    const unsigned int lt = (1u << lane) - 1u;
    const int my_gt = gt_before + run_gt + __popc(bg & lt);
    const int my_eq = eq_before + run_eq + __popc(be & lt);
    if (gt || (eq && my_eq < need_eq)) {
      const int pos = my_gt + min(my_eq, need_eq);
      if (pos < rd.k) out[pos] = j;
    }
    run_gt += __popc(bg);
    run_eq += __popc(be);
  }
  for (int j = rd.k + tid; j < a.k_stride; j += kThreads) out[j] = -1;
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  size_t smem = (2048 + 2 * kCandCap) * sizeof(uint32_t);
  if (a.n <= kRowCap) smem += static_cast<size_t>(a.n) * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k_topk<<<a.rows, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace kascade
