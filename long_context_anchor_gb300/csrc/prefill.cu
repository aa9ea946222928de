// prefill.cu — tiled causal prefill on the tcgen05 tensor cores (Kascade
// prefill works at tile level; opentrain.ai Abstract "tile-level operations";
// one index set per (head, 128-query tile)).
//
//   k_prefill_fa<REUSE, LSE>  one CTA per (sequence, query head, 128-row tile):
//       a TMA producer warp streams the Q tile and 128-key K/V tiles (dense:
//       key tiles 0..t, causal; reuse: the tile's saved keys, gathered four
//       rows per TMA tile::gather4), one thread issues tcgen05.mma
//       S = Q K^T into double-buffered TMEM and O += P V, and a softmax
//       warpgroup (one thread per query row) runs the online softmax with a
//       lazy O rescale (only when a row maximum grows by more than 2^8),
//       writes P as bf16 to shared memory and finally O / l (and, for anchor
//       layers, the row log-sum-exp). Causal masking is by key position.
//   k_prefill_weights        anchor pass 2: S^T = K Q^T per key tile (TMEM lane
//       = key), p = 2^(s*sigma*log2e - lse2[query]), and each thread sums its
//       key's column over the tile's rows: w_j = sum_{i in tile, i >= j} p_ij,
//       written to the packed tile-weight rows that the Top-k reads.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace kascade {
namespace {

constexpr int kTile = 128;              // query rows and keys per tile
constexpr int kHalf = kTile * 128;      // bytes of one 64-column half of a tile
constexpr int kTileBytes = 2 * kHalf;   // 128 x 128 bf16 = 32 KB
constexpr int kFaThreads = 256;         // warp 0 TMA, warp 1 MMA, warps 4-7 softmax
constexpr float kRescaleLog2 = 8.0f;    // lazy O rescale threshold (factor 256)
#define kNegInfP (-CUDART_INF_F)

struct FaSmem {
  // 1024-aligned tile region (offsets from the aligned base)
  static constexpr int Q = 0;
  static constexpr int K0 = Q + kTileBytes;          // K[2]
  static constexpr int V0 = K0 + 2 * kTileBytes;     // V[2]
  static constexpr int P = V0 + 2 * kTileBytes;
  static constexpr int POS = P + kTileBytes;         // int32 [2][128] key positions
  static constexpr int BAR = POS + 2 * kTile * 4;    // mbarriers
  static constexpr int TMEM = BAR + 16 * 8;
  static constexpr int BYTES = TMEM + 16;
};
constexpr size_t kFaSmemBytes = FaSmem::BYTES + 1024;

// tcgen05 descriptors of the 128x128 tiles (see tc.cuh).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
  return sw128_desc(tile + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t vmn_desc(uint32_t tile, int kk) {
  return sw128_desc(tile + kk * 2048, kHalf, 1024);
}

// Work order: longest tiles (largest t) first.
__device__ __forceinline__ void fa_tile_coords(const PrefillArgs& a, int& bh, int& t) {
  const int BH = a.B * a.Hq;
  bh = blockIdx.x % BH;
  t = a.nT - 1 - static_cast<int>(blockIdx.x) / BH;
}

template <bool REUSE, bool LSE>
__global__ void __launch_bounds__(kFaThreads, 1)
    k_prefill_fa(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ PrefillArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int32_t* s_pos = reinterpret_cast<int32_t*>(sm + FaSmem::POS);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + FaSmem::BAR);
  uint64_t* q_full = bar + 0;
  uint64_t* kv_full = bar + 1;   // [2]
  uint64_t* kv_free = bar + 3;   // [2]
  uint64_t* s_full = bar + 5;    // [2]
  uint64_t* s_free = bar + 7;    // [2]
  uint64_t* p_full = bar + 9;
  uint64_t* pv_done = bar + 10;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + FaSmem::TMEM);
  const uint32_t sQ = smem_u32(sm + FaSmem::Q), sK0 = smem_u32(sm + FaSmem::K0);
  const uint32_t sV0 = smem_u32(sm + FaSmem::V0), sP = smem_u32(sm + FaSmem::P);

  int bh, t;
  fa_tile_coords(a, bh, t);
  const int b = bh / a.Hq, h = bh % a.Hq, g = a.head_kv[h];
  const int row0 = t * kTile;
  const int L = min(a.N, row0 + kTile);   // causal prefix of the tile
  int nkv, kt = 0;
  const int32_t* idx_row = nullptr;
  if (REUSE) {
    kt = min(a.topk, L);
    nkv = (kt + kTile - 1) / kTile;
    idx_row = a.idx + (static_cast<size_t>(bh) * a.nT + t) * a.topk;
  } else {
    nkv = (L + kTile - 1) / kTile;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(kv_full + s, 1);
      mbar_init(kv_free + s, 1);
      mbar_init(s_full + s, 1);
      mbar_init(s_free + s, 128);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    fence_barrier_init();
  }
  if (warp == 2) tmem_alloc(s_tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t tS = tmem, tO = tmem + 256;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    const int kv_row_base = (b * a.Hkv + g) * a.N;
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_2d(sm + FaSmem::Q, &tmQ, q_full, 0, bh * a.N + row0);
      tma_load_2d(sm + FaSmem::Q + kHalf, &tmQ, q_full, 64, bh * a.N + row0);
    }
    int issued = 0;
    for (int j = 0; j < nkv; ++j) {
      const int s = j & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(kv_free + s, ((j >> 1) & 1) ^ 1, a.err, 0x601);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      unsigned char* kd = sm + FaSmem::K0 + s * kTileBytes;
      unsigned char* vd = sm + FaSmem::V0 + s * kTileBytes;
      if (!REUSE) {
        if (lane == 0) {
          mbar_arrive_expect_tx(kv_full + s, 2 * kTileBytes);
          const int y = kv_row_base + j * kTile;
          tma_load_2d(kd, &tmK, kv_full + s, 0, y);
          tma_load_2d(kd + kHalf, &tmK, kv_full + s, 64, y);
          tma_load_2d(vd, &tmV, kv_full + s, 0, y);
          tma_load_2d(vd + kHalf, &tmV, kv_full + s, 64, y);
        }
      } else {
        // Padding slots (and invalid entries) gather the tile's first saved
        // row, which is selected anyway, and are masked in the softmax; rows
        // outside the saved set are never read.
        int p_first = __ldg(idx_row);
        if (p_first < 0 || p_first >= a.N) p_first = 0;
        int rows[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = j * kTile + lane * 4 + u;
          int p = e < kt ? __ldg(idx_row + e) : -1;
          if (p >= a.N || (e < kt && p < 0)) {
            report_error(a.err, KASCADE_ERR_BAD_INPUT, 0x602);
            p = -1;
          }
          s_pos[s * kTile + lane * 4 + u] = p;
          rows[u] = kv_row_base + (p >= 0 ? p : p_first);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(kv_full + s, 2 * kTileBytes);
        __syncwarp();
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          tma_gather4(kd + hf * kHalf + lane * 512, &tmK, kv_full + s, hf * 64, rows[0], rows[1],
                      rows[2], rows[3]);
          tma_gather4(vd + hf * kHalf + lane * 512, &tmV, kv_full + s, hf * 64, rows[0], rows[1],
                      rows[2], rows[3]);
        }
      }
      issued = j + 1;
    }
    // Never leave with copies in flight.
    if (lane == 0) {
      mbar_wait(q_full, 0, a.err, 0x603);
      for (int j = issued > 2 ? issued - 2 : 0; j < issued; ++j)
        mbar_wait(kv_full + (j & 1), (j >> 1) & 1, a.err, 0x604);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idq = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idv = idesc_bf16_f32(128, 128, 0, 1);
      bool ok = mbar_wait(q_full, 0, a.err, 0x611);
      auto issue_pv = [&](int jj) {
        const int s = jj & 1;
        if (!mbar_wait(p_full, jj & 1, a.err, 0x612)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma(tO, kmajor_desc(sP, kk), vmn_desc(sV0 + s * kTileBytes, kk), idv,
                 (jj > 0 || kk > 0) ? 1u : 0u);
        tc_commit(pv_done);
        tc_commit(kv_free + s);
        return true;
      };
      for (int j = 0; ok && j < nkv; ++j) {
        const int s = j & 1;
        ok = mbar_wait(kv_full + s, (j >> 1) & 1, a.err, 0x613) &&
             mbar_wait(s_free + s, ((j >> 1) & 1) ^ 1, a.err, 0x614);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma(tS + s * 128, kmajor_desc(sQ, kk), kmajor_desc(sK0 + s * kTileBytes, kk), idq,
                 kk > 0 ? 1u : 0u);
        tc_commit(s_full + s);
        if (j > 0) ok = issue_pv(j - 1);
      }
      if (ok && nkv > 0) issue_pv(nkv - 1);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax warpgroup
    const int r = (warp - 4) * 32 + lane;
    const int i = row0 + r;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float m_used = kNegInfP, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int s = j & 1;
      ok = mbar_wait(s_full + s, (j >> 1) & 1, a.err, 0x621);
      if (!ok) break;
      tc_fence_after();
      float x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tS + s * 128 + c * 32 + lane_base, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(v[e]);
      }
      tc_fence_before();
      mbar_arrive(s_free + s);
      float tmax = kNegInfP;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        const int kp = REUSE ? s_pos[s * kTile + c] : j * kTile + c;
        const bool valid = kp >= 0 && kp <= i;
        x[c] = valid ? x[c] * a.scale_log2 : kNegInfP;
        tmax = fmaxf(tmax, x[c]);
      }
      float alpha = 1.f;
      bool resc = false;
      if (tmax > m_used + kRescaleLog2) {
        if (j > 0) {
          alpha = ex2_approx(m_used - tmax);   // 0 when m_used = -inf
          resc = true;
        }
        l *= alpha;
        m_used = tmax;
      }
      const float mu = (m_used == kNegInfP) ? 0.f : m_used;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = ex2_approx(x[2 * c] - mu), p1 = ex2_approx(x[2 * c + 1] - mu);
        l += p0 + p1;
        pk[c] = pack_bf16(p0, p1);
      }
      if (j > 0) {
        ok = mbar_wait(pv_done, (j - 1) & 1, a.err, 0x622);
        if (!ok) break;
      }
      if (__any_sync(0xffffffffu, resc)) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32 + lane_base, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + c * 32 + lane_base, o);
        }
        tmem_wait_st();
      }
      // P row -> shared memory, K-major 128-byte-swizzled (A operand of P V)
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        const uint32_t addr =
            sP + (ch >> 3) * kHalf + r * 128 + ((((ch & 7) ^ (r & 7))) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(pk[4 * ch]),
                     "r"(pk[4 * ch + 1]), "r"(pk[4 * ch + 2]), "r"(pk[4 * ch + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    // epilogue: O / l -> bf16 row; anchor layers also keep the row LSE (log2 units)
    if (ok && nkv > 0) ok = mbar_wait(pv_done, (nkv - 1) & 1, a.err, 0x623);
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16* orow =
        static_cast<__nv_bfloat16*>(a.out) + (static_cast<size_t>(bh) * a.N + i) * kTile;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      tmem_ld32(tO + c * 32 + lane_base, o);
      tmem_wait_ld();
      uint32_t ob[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        ob[e] = (nkv > 0 && ok) ? pack_bf16(__uint_as_float(o[2 * e]) * inv,
                                            __uint_as_float(o[2 * e + 1]) * inv)
                                : 0u;
      if (i < a.N) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(ob[4 * q], ob[4 * q + 1], ob[4 * q + 2], ob[4 * q + 3]);
      }
    }
    if (LSE && i < a.N)
      a.lse[static_cast<size_t>(bh) * a.N + i] = l > 0.f ? m_used + __log2f(l) : kNegInfP;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------
// Anchor pass 2: tile weights from S^T = K_j Q_t^T (TMEM lane = key).
// ------------------------------------------------------------------------
struct WtSmem {
  static constexpr int Q = 0;
  static constexpr int K0 = Q + kTileBytes;      // K[2]
  static constexpr int LSE = K0 + 2 * kTileBytes;  // float [128]
  static constexpr int BAR = LSE + kTile * 4;
  static constexpr int TMEM = BAR + 16 * 8;
  static constexpr int BYTES = TMEM + 16;
};
constexpr size_t kWtSmemBytes = WtSmem::BYTES + 1024;

__global__ void __launch_bounds__(kFaThreads, 1)
    k_prefill_weights(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK, const __grid_constant__ PrefillArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* s_lse = reinterpret_cast<float*>(sm + WtSmem::LSE);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + WtSmem::BAR);
  uint64_t* q_full = bar + 0;
  uint64_t* k_full = bar + 1;   // [2]
  uint64_t* k_free = bar + 3;   // [2]
  uint64_t* s_full = bar + 5;   // [2]
  uint64_t* s_free = bar + 7;   // [2]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + WtSmem::TMEM);
  const uint32_t sQ = smem_u32(sm + WtSmem::Q), sK0 = smem_u32(sm + WtSmem::K0);

  int bh, t;
  fa_tile_coords(a, bh, t);
  const int b = bh / a.Hq, h = bh % a.Hq, g = a.head_kv[h];
  const int row0 = t * kTile;
  const int L = min(a.N, row0 + kTile);
  const int nkv = (L + kTile - 1) / kTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_free + s, 1);
      mbar_init(s_full + s, 1);
      mbar_init(s_free + s, 128);
    }
    fence_barrier_init();
  }
  if (warp >= 4) {
    const int r = threadIdx.x - 128;
    const int i = row0 + r;
    s_lse[r] = i < a.N ? a.lse[static_cast<size_t>(bh) * a.N + i] : CUDART_INF_F;
  }
  if (warp == 2) tmem_alloc(s_tmem, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      const int kv_row_base = (b * a.Hkv + g) * a.N;
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_2d(sm + WtSmem::Q, &tmQ, q_full, 0, bh * a.N + row0);
      tma_load_2d(sm + WtSmem::Q + kHalf, &tmQ, q_full, 64, bh * a.N + row0);
      int issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int s = j & 1;
        if (!mbar_wait(k_free + s, ((j >> 1) & 1) ^ 1, a.err, 0x701)) break;
        unsigned char* kd = sm + WtSmem::K0 + s * kTileBytes;
        mbar_arrive_expect_tx(k_full + s, kTileBytes);
        tma_load_2d(kd, &tmK, k_full + s, 0, kv_row_base + j * kTile);
        tma_load_2d(kd + kHalf, &tmK, k_full + s, 64, kv_row_base + j * kTile);
        issued = j + 1;
      }
      mbar_wait(q_full, 0, a.err, 0x702);
      for (int j = issued > 2 ? issued - 2 : 0; j < issued; ++j)
        mbar_wait(k_full + (j & 1), (j >> 1) & 1, a.err, 0x703);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id = idesc_bf16_f32(128, 128, 0, 0);
      bool ok = mbar_wait(q_full, 0, a.err, 0x711);
      for (int j = 0; ok && j < nkv; ++j) {
        const int s = j & 1;
        ok = mbar_wait(k_full + s, (j >> 1) & 1, a.err, 0x712) &&
             mbar_wait(s_free + s, ((j >> 1) & 1) ^ 1, a.err, 0x713);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma(tmem + s * 128, kmajor_desc(sK0 + s * kTileBytes, kk), kmajor_desc(sQ, kk), id,
                 kk > 0 ? 1u : 0u);
        tc_commit(s_full + s);
        tc_commit(k_free + s);
      }
    }
  } else if (warp >= 4) {
    const int r = threadIdx.x - 128;   // key lane within the key tile
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float* wrow = a.w + static_cast<size_t>(bh) * (static_cast<size_t>(64) * (a.nT - 1) * a.nT + a.N) +
                  static_cast<size_t>(64) * t * (t + 1);
    for (int j = 0; j < nkv; ++j) {
      const int s = j & 1;
      if (!mbar_wait(s_full + s, (j >> 1) & 1, a.err, 0x721)) break;
      tc_fence_after();
      const int kj = j * kTile + r;
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + s * 128 + c * 32 + lane_base, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int q = c * 32 + e;
          const float p = ex2_approx(__uint_as_float(v[e]) * a.scale_log2 - s_lse[q]);
          sum += (kj <= row0 + q) ? p : 0.f;
        }
      }
      tc_fence_before();
      mbar_arrive(s_free + s);
      if (kj < L) wrow[kj] = sum;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

bool make_maps(const PrefillArgs& a, CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv,
               bool gather) {
  const uint64_t qrows = static_cast<uint64_t>(a.B) * a.Hq * a.N;
  const uint64_t kvrows = static_cast<uint64_t>(a.B) * a.Hkv * a.N;
  if (tq && !encode_tmap_2d_bf16(tq, a.q, 128, qrows, 64, kTile, true)) return false;
  const uint32_t box_rows = gather ? 1 : kTile;
  if (tk && !encode_tmap_2d_bf16(tk, a.k, 128, kvrows, 64, box_rows, true)) return false;
  if (tv && !encode_tmap_2d_bf16(tv, a.v, 128, kvrows, 64, box_rows, true)) return false;
  return true;
}

template <bool REUSE, bool LSE>
cudaError_t launch_fa(const PrefillArgs& a, cudaStream_t st) {
  alignas(64) CUtensorMap tq, tk, tv;
  if (!make_maps(a, &tq, &tk, &tv, REUSE)) return cudaErrorInvalidValue;
  auto kern = k_prefill_fa<REUSE, LSE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kFaSmemBytes));
  if (e != cudaSuccess) return e;
  kern<<<a.B * a.Hq * a.nT, kFaThreads, kFaSmemBytes, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_dense(const PrefillArgs& a, int head_dim, cudaStream_t st) {
  if (head_dim != 128) return cudaErrorNotSupported;
  return launch_fa<false, false>(a, st);
}

cudaError_t launch_prefill_lse(const PrefillArgs& a, int head_dim, cudaStream_t st) {
  if (head_dim != 128) return cudaErrorNotSupported;
  return launch_fa<false, true>(a, st);   // exact output + row LSE
}

cudaError_t launch_prefill_anchor_main(const PrefillArgs& a, int head_dim, cudaStream_t st) {
  if (head_dim != 128) return cudaErrorNotSupported;
  alignas(64) CUtensorMap tq, tk;
  if (!make_maps(a, &tq, &tk, nullptr, false)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k_prefill_weights,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kWtSmemBytes));
  if (e != cudaSuccess) return e;
  k_prefill_weights<<<a.B * a.Hq * a.nT, kFaThreads, kWtSmemBytes, st>>>(tq, tk, a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_reuse(const PrefillArgs& a, int head_dim, cudaStream_t st) {
  if (head_dim != 128) return cudaErrorNotSupported;
  return launch_fa<true, false>(a, st);
}

}  // namespace kascade
