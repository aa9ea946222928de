// prefill.cu — tiled causal prefill on the tcgen05 tensor cores (Kascade
// prefill works at tile level; opentrain.ai Abstract "tile-level operations";
// one index set per (head, 128-query tile)).
//
//   k_prefill_fa<REUSE, LSE>  one CTA per (sequence, query head, 128-row tile):
//       a TMA producer warp streams the Q tile and, for dense/anchor layers,
//       the causal 128-key K/V tiles 0..t; for reuse layers two warps gather
//       the tile's saved K/V rows in 64-key chunks (16-byte cp.async into the
//       128-byte-swizzled layout, four chunks in flight, then
//       fence.proxy.async before signalling the MMA); one thread issues tcgen05.mma
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

// Shared-memory plan of k_prefill_fa for KC-key chunks and an ST-deep K/V ring.
template <int KC, int ST>
struct FaCfg {
  static constexpr int KHALF = KC * 128;          // one 64-dim half of a K (or V) chunk
  static constexpr int KV_BYTES = 2 * KHALF;      // one K (or V) chunk, 128 dims
  static constexpr int P_BYTES = kTile * KC * 2;  // P tile, bf16
  static constexpr int Q = 0;
  static constexpr int K0 = Q + kTileBytes;
  static constexpr int V0 = K0 + ST * KV_BYTES;
  static constexpr int P = V0 + ST * KV_BYTES;
  static constexpr int POS = P + P_BYTES;          // int32 [ST][KC] key positions
  static constexpr int BAR = POS + ST * KC * 4;
  static constexpr int TMEM = BAR + 32 * 8;
  static constexpr int BYTES = TMEM + 16;
  static constexpr size_t SMEM = BYTES + 1024;
};

// tcgen05 descriptors (see tc.cuh): K-major tiles with `half` bytes per
// 64-column half; V as an MN-major B operand with `half` bytes per 64 dims.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk, int half = kHalf) {
  return sw128_desc(tile + (kk >> 2) * half + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t vmn_desc(uint32_t tile, int kk, int half = kHalf) {
  return sw128_desc(tile + kk * 2048, half, 1024);
}

// Work order: longest tiles (largest t) first.
__device__ __forceinline__ void fa_tile_coords(const PrefillArgs& a, int& bh, int& t) {
  const int BH = a.B * a.Hq;
  bh = blockIdx.x % BH;
  t = a.nT - 1 - static_cast<int>(blockIdx.x) / BH;
}

// REUSE: keys come from the tile's saved set (gathered by warps 2-3 with
// 16-byte cp.async into the swizzled layout, then fence.proxy.async);
// otherwise the causal key tiles 0..t stream in by TMA (warp 0).
// LSE: also store the row log-sum-exp (log2 units) for the tile weights.
template <bool REUSE, bool LSE, int KC, int ST>
__global__ void __launch_bounds__(kFaThreads, 1)
    k_prefill_fa(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ PrefillArgs a) {
  using C = FaCfg<KC, ST>;
  constexpr int LA = ST / 2;   // cp.async chunks kept in flight before signalling
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int32_t* s_pos = reinterpret_cast<int32_t*>(sm + C::POS);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + C::BAR);
  uint64_t* q_full = bar + 0;
  uint64_t* kv_full = bar + 1;          // [ST]
  uint64_t* kv_free = bar + 1 + ST;     // [ST]
  uint64_t* s_full = bar + 1 + 2 * ST;  // [2]
  uint64_t* s_free = s_full + 2;        // [2]
  uint64_t* p_full = s_free + 2;
  uint64_t* pv_done = p_full + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + C::TMEM);
  const uint32_t sQ = smem_u32(sm + C::Q), sK0 = smem_u32(sm + C::K0);
  const uint32_t sV0 = smem_u32(sm + C::V0), sP = smem_u32(sm + C::P);

  int bh, t;
  fa_tile_coords(a, bh, t);
  const int b = bh / a.Hq, h = bh % a.Hq, g = a.head_kv[h];
  const int row0 = t * kTile;
  const int L = min(a.N, row0 + kTile);   // causal prefix of the tile
  int nkv, kt = 0;
  const int32_t* idx_row = nullptr;
  if (REUSE) {
    kt = min(a.topk, L);
    nkv = (kt + KC - 1) / KC;
    idx_row = a.idx + (static_cast<size_t>(bh) * a.nT + t) * a.topk;
  } else {
    nkv = (L + KC - 1) / KC;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kv_row_base = (b * a.Hkv + g) * a.N;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(kv_full + s, REUSE ? 64 : 1);
      mbar_init(kv_free + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
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
    // ------------------------------------------------ TMA: Q, and dense K/V
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_2d(sm + C::Q, &tmQ, q_full, 0, bh * a.N + row0);
      tma_load_2d(sm + C::Q + kHalf, &tmQ, q_full, 64, bh * a.N + row0);
      if (!REUSE) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        int issued = 0;
        for (int j = 0; j < nkv; ++j) {
          const int s = j % ST;
          if (!mbar_wait(kv_free + s, ((j / ST) & 1) ^ 1, a.err, 0x601)) break;
          unsigned char* kd = sm + C::K0 + s * C::KV_BYTES;
          unsigned char* vd = sm + C::V0 + s * C::KV_BYTES;
          mbar_arrive_expect_tx(kv_full + s, 2 * C::KV_BYTES);
          const int y = kv_row_base + j * KC;
          tma_load_2d(kd, &tmK, kv_full + s, 0, y);
          tma_load_2d(kd + C::KHALF, &tmK, kv_full + s, 64, y);
          tma_load_2d(vd, &tmV, kv_full + s, 0, y);
          tma_load_2d(vd + C::KHALF, &tmV, kv_full + s, 64, y);
          issued = j + 1;
        }
        for (int j = issued > ST ? issued - ST : 0; j < issued; ++j)
          mbar_wait(kv_full + (j % ST), (j / ST) & 1, a.err, 0x604);
      }
      mbar_wait(q_full, 0, a.err, 0x603);   // never leave with copies in flight
    }
  } else if (REUSE && (warp == 2 || warp == 3)) {
    // ------------------------------------------------ gather producer (64 threads, one key row each)
    static_assert(!REUSE || KC == 64, "one gathered row per producer thread");
    const int pt = threadIdx.x - 64;
    int p_first = __ldg(idx_row);
    if (p_first < 0 || p_first >= a.N) p_first = 0;
    const __nv_bfloat16* kbase = static_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* vbase = static_cast<const __nv_bfloat16*>(a.v);
    int issued = 0;
    for (int j = 0; j < nkv; ++j) {
      const int s = j % ST;
      if (!mbar_wait(kv_free + s, ((j / ST) & 1) ^ 1, a.err, 0x605)) break;
      const int e = j * KC + pt;
      int p = e < kt ? __ldg(idx_row + e) : -1;
      if (p >= a.N || (e < kt && p < 0)) {
        report_error(a.err, KASCADE_ERR_BAD_INPUT, 0x602);
        p = -1;
      }
      s_pos[s * KC + pt] = p;
      // padding slots re-read the tile's first saved row (masked later)
      const size_t row = static_cast<size_t>(kv_row_base) + (p >= 0 ? p : p_first);
      const __nv_bfloat16* ks = kbase + row * 128;
      const __nv_bfloat16* vs = vbase + row * 128;
      unsigned char* kd = sm + C::K0 + s * C::KV_BYTES;
      unsigned char* vd = sm + C::V0 + s * C::KV_BYTES;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int off = (c >> 3) * C::KHALF + pt * 128 + (((c & 7) ^ (pt & 7)) << 4);
        cp_async16(kd + off, ks + c * 8, 16);
        cp_async16(vd + off, vs + c * 8, 16);
      }
      cp_async_commit();
      issued = j + 1;
      if (j >= LA) {
        cp_async_wait<LA>();
        fence_proxy_async_smem();
        mbar_arrive(kv_full + (j - LA) % ST);
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    for (int j = issued > LA ? issued - LA : 0; j < issued; ++j) mbar_arrive(kv_full + j % ST);
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idq = idesc_bf16_f32(128, KC, 0, 0);
      constexpr uint32_t idv = idesc_bf16_f32(128, 128, 0, 1);
      bool ok = mbar_wait(q_full, 0, a.err, 0x611);
      auto issue_pv = [&](int jj) {
        const int s = jj % ST;
        if (!mbar_wait(p_full, jj & 1, a.err, 0x612)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < KC / 16; ++kk)
          tc_mma(tO, kmajor_desc(sP, kk), vmn_desc(sV0 + s * C::KV_BYTES, kk, C::KHALF), idv,
                 (jj > 0 || kk > 0) ? 1u : 0u);
        tc_commit(pv_done);
        tc_commit(kv_free + s);
        return true;
      };
      for (int j = 0; ok && j < nkv; ++j) {
        const int s = j % ST, sb = j & 1;
        ok = mbar_wait(kv_full + s, (j / ST) & 1, a.err, 0x613) &&
             mbar_wait(s_free + sb, ((j >> 1) & 1) ^ 1, a.err, 0x614);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma(tS + sb * 128, kmajor_desc(sQ, kk),
                 kmajor_desc(sK0 + s * C::KV_BYTES, kk, C::KHALF), idq, kk > 0 ? 1u : 0u);
        tc_commit(s_full + sb);
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
      const int sb = j & 1, s = j % ST;
      ok = mbar_wait(s_full + sb, (j >> 1) & 1, a.err, 0x621);
      if (!ok) break;
      tc_fence_after();
      float x[KC];
#pragma unroll
      for (int c = 0; c < KC / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tS + sb * 128 + c * 32 + lane_base, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(v[e]);
      }
      tc_fence_before();
      mbar_arrive(s_free + sb);
      // raw-score maximum; the causal mask is needed only where keys can
      // exceed this row (dense: the diagonal tile; reuse: every chunk)
      const bool need_mask = REUSE || (j * KC + KC - 1 > row0);
      float tmax = kNegInfP;
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < KC; ++c) {
          const int kp = REUSE ? s_pos[s * KC + c] : j * KC + c;
          if (!(kp >= 0 && kp <= i)) x[c] = kNegInfP;
          tmax = fmaxf(tmax, x[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < KC; ++c) tmax = fmaxf(tmax, x[c]);
      }
      tmax *= a.scale_log2;   // scale > 0: max commutes with scaling
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
      uint32_t pk[KC / 2];
#pragma unroll
      for (int c = 0; c < KC / 2; ++c) {
        const float p0 = ex2_approx(fmaf(x[2 * c], a.scale_log2, -mu));
        const float p1 = ex2_approx(fmaf(x[2 * c + 1], a.scale_log2, -mu));
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
      for (int ch = 0; ch < KC / 8; ++ch) {
        const uint32_t addr = sP + (ch >> 3) * kHalf + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
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

// Q tiles of 128 rows; K/V tiles of kv_rows rows (2-D maps over all heads).
bool make_maps(const PrefillArgs& a, CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv,
               int kv_rows) {
  const uint64_t qrows = static_cast<uint64_t>(a.B) * a.Hq * a.N;
  const uint64_t kvrows = static_cast<uint64_t>(a.B) * a.Hkv * a.N;
  if (tq && !encode_tmap_2d_bf16(tq, a.q, 128, qrows, 64, kTile, true)) return false;
  if (tk && !encode_tmap_2d_bf16(tk, a.k, 128, kvrows, 64, kv_rows, true)) return false;
  if (tv && !encode_tmap_2d_bf16(tv, a.v, 128, kvrows, 64, kv_rows, true)) return false;
  return true;
}

template <bool REUSE, bool LSE, int KC, int ST>
cudaError_t launch_fa(const PrefillArgs& a, cudaStream_t st) {
  alignas(64) CUtensorMap tq, tk, tv;
  if (!make_maps(a, &tq, &tk, &tv, KC)) return cudaErrorInvalidValue;
  auto kern = k_prefill_fa<REUSE, LSE, KC, ST>;
  const size_t smem = FaCfg<KC, ST>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<a.B * a.Hq * a.nT, kFaThreads, smem, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_dense(const PrefillArgs& a, int head_dim, cudaStream_t st) {
  if (head_dim != 128) return cudaErrorNotSupported;
  return launch_fa<false, false, 128, 2>(a, st);
}

cudaError_t launch_prefill_lse(const PrefillArgs& a, int head_dim, cudaStream_t st) {
  if (head_dim != 128) return cudaErrorNotSupported;
  return launch_fa<false, true, 128, 2>(a, st);   // exact output + row LSE
}

cudaError_t launch_prefill_anchor_main(const PrefillArgs& a, int head_dim, cudaStream_t st) {
  if (head_dim != 128) return cudaErrorNotSupported;
  alignas(64) CUtensorMap tq, tk;
  if (!make_maps(a, &tq, &tk, nullptr, kTile)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k_prefill_weights,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kWtSmemBytes));
  if (e != cudaSuccess) return e;
  k_prefill_weights<<<a.B * a.Hq * a.nT, kFaThreads, kWtSmemBytes, st>>>(tq, tk, a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_reuse(const PrefillArgs& a, int head_dim, cudaStream_t st) {
  if (head_dim != 128) return cudaErrorNotSupported;
  return launch_fa<true, false, 64, 4>(a, st);
}

}  // namespace kascade
