// prefill.cu — tiled causal prefill on the tcgen05 tensor cores (Kascade
// prefill works at tile level; opentrain.ai Abstract "tile-level operations";
// one index set per (head, 128-query tile)).
//
//   k_prefill_fa2<REUSE, LSE>  persistent, one CTA per SM taking (sequence,
//       query head, 128-row) tiles in turn; a tile's 64-key chunks are split
//       over two pipelines that share the Q tile and merge their partial
//       softmax states at the end: a loader warp brings the Q tiles by TMA and
//       producer warps the keys (dense/anchor layers: causal K/V tiles by TMA;
//       reuse layers: the tile's saved K/V rows by coalesced 16-byte cp.async
//       into the 128-byte-swizzled layout, then fence.proxy.async), running
//       ahead into the next tile; Q is copied into TMEM and is the A operand
//       of every S = Q K^T; one warp per pipeline issues tcgen05.mma S = Q K^T
//       and O += P V with P read from TMEM; a softmax warpgroup per pipeline
//       (one thread per query row) runs the online softmax with a lazy O
//       rescale (only when a row maximum grows by more than 2^8) and writes P
//       as bf16 into TMEM; at the end of a tile both pipelines merge the two
//       partial states (half the output dims each) and write O / l (and, for
//       anchor layers, the row log-sum-exp). Causal masking is by key
//       position.
//   k_prefill_weights        anchor pass 2, persistent like the kernel above:
//       S^T = K Q^T per key tile (TMEM lane = key), p = 2^(s*sigma*log2e -
//       lse2[query]), and each thread sums its key's column over the tile's
//       rows: w_j = sum_{i in tile, i >= j} p_ij, written to the packed
//       tile-weight rows that the Top-k reads.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace kascade {
namespace {

template <bool V>
struct BoolC {
  static constexpr bool value = V;
};

constexpr int kTile = 128;              // query rows and keys per tile
constexpr int kHalf = kTile * 128;      // bytes of one 64-column half of a tile
constexpr int kTileBytes = 2 * kHalf;   // 128 x 128 bf16 = 32 KB
constexpr int kWtGroups = 3;            // weights kernel: epilogue warpgroups
constexpr int kWtThreads = 128 + 128 * kWtGroups;   // warp 0 TMA, warp 1 MMA, warps 4.. epilogue
constexpr float kRescaleLog2 = 8.0f;    // lazy O rescale threshold (factor 256)
#define kNegInfP (-CUDART_INF_F)

// tcgen05 descriptors (see tc.cuh): K-major tiles with `half` bytes per
// 64-column half; V as an MN-major B operand with `half` bytes per 64 dims.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk, int half = kHalf) {
  return sw128_desc(tile + (kk >> 2) * half + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t vmn_desc(uint32_t tile, int kk, int half = kHalf) {
  return sw128_desc(tile + kk * 2048, half, 1024);
}

// Persistent tiles: one CTA per SM takes the query tiles tau = blockIdx.x,
// blockIdx.x + gridDim.x, ... (longest tiles first), each tile's 64-key chunks
// split over two pipelines (pipe p takes chunks p, p+2, ...) that share the Q
// tile and merge their partial softmax states at the end of the tile. Every
// barrier phase and ring stage runs on per-pipeline chunk counters that carry
// over from tile to tile, so the producers stream the next tile's chunks and
// a dedicated warp loads its Q tile while the current tile is still being
// computed; a tile boundary costs only the merge and the copy of the next Q
// into TMEM.
// Roles: warps 4p..4p+3 run pipe p's softmax, warp 8+p issues its MMAs, warp
// 10+p is its producer (dense: TMA; reuse: warps 10+p and 12+p gather its
// chunks in turn with coalesced 16-byte cp.async, two chunks in flight each),
// and the last warp loads the Q tiles by TMA.
// The Q tile is copied once into TMEM, where it is the A operand of every
// S = Q K^T of both pipes, so shared memory feeds only K and V to the tensor
// core. Every pipe has an ST-deep K/V ring in shared memory and its own score,
// P and O columns in TMEM: the softmax releases the scores as soon as it has
// read them (so S of the next chunk overlaps its exponentials), writes P as
// bf16 into the P columns once the previous P V product has landed, and the
// P V product takes P from TMEM as its A operand, so P never touches shared
// memory. At the end of a tile pipe 1 hands its (m, l) to pipe 0 through its
// own (then idle) P columns; pipe 0 copies the next Q into TMEM, so the next
// tile's first scores overlap the merge, then reads both O accumulators.
template <bool REUSE> __host__ __device__ constexpr int fa_threads() { return REUSE ? 480 : 416; }
template <bool REUSE> __host__ __device__ constexpr int fa_q_warp() { return REUSE ? 14 : 12; }

// Chunk shape: KC keys per chunk and an ST-deep K/V ring per pipeline; the same
// for streamed (TMA) and gathered chunks.
template <bool REUSE> struct FaShape { static constexpr int KC = 64, ST = 3; };

template <bool REUSE>
struct Fa2Smem {
  static constexpr int KC = FaShape<REUSE>::KC, ST = FaShape<REUSE>::ST;
  static constexpr int KHALF = KC * 128;             // one 64-dim half of a K (or V) chunk
  static constexpr int KV_BYTES = 2 * KHALF;
  static constexpr int K0 = 0;                       // within a pipeline's area
  static constexpr int V0 = ST * KV_BYTES;
  static constexpr int PIPE_BYTES = 2 * ST * KV_BYTES;
  static constexpr int Q = 0;                        // Q staging (TMA target)
  static constexpr int PIPE0 = kTileBytes;
  static constexpr int PIPE1 = PIPE0 + PIPE_BYTES;
  static constexpr int POS = PIPE1 + PIPE_BYTES;     // reuse: int32 [2 pipes][ST][KC] + flags [2][ST]
  static constexpr int POS_BYTES = REUSE ? 2 * ST * (KC + 1) * 4 : 0;
  static constexpr int NB = 2 * ST + 4;             // mbarriers per pipeline
  static constexpr int BAR = POS + POS_BYTES;        // [2 pipes][NB] + q_full + q_ready
  static constexpr int TMEM = BAR + (2 * NB + 4) * 8;   // + q_full, q_ready, o_ready[2]
  static constexpr int BYTES = TMEM + 8;
  static constexpr size_t SMEM = BYTES + 1024;       // + slack for 1024-byte alignment
  static_assert(SMEM <= 232448, "the tile and two pipelines must fit in shared memory");
  // TMEM columns: Q (bf16 pairs) [0, 64); pipeline p at 64 + 224 p: scores S
  // (KC fp32 columns), P (KC / 2 columns of bf16 pairs), O (128 columns)
  static constexpr int T_PIPE = 64, T_PIPE_COLS = 224;
  static constexpr int T_S = 0, T_P = 64, T_O = 96;
  static_assert(KC <= 64 && T_O + 128 == T_PIPE_COLS, "pipeline TMEM columns");
  static_assert(T_PIPE + 2 * T_PIPE_COLS == 512, "TMEM holds Q and two pipelines");
  static_assert(KC % 32 == 0 && KC <= 64, "softmax reads scores 32 columns at a time");
};

// P (KC bf16 per row, packed in pairs) into KC/2 TMEM columns of this warp's lanes.
template <int KC>
__device__ __forceinline__ void tmem_store_p(uint32_t taddr, const uint32_t (&pk)[KC / 2]) {
  if constexpr (KC == 64) {
    tmem_st32(taddr, pk);
  } else {
    static_assert(KC == 32, "P chunks are 32 or 64 keys");
    tmem_st16(taddr, pk);
  }
}

// One query tile of the persistent schedule.
struct FaTile {
  int bh, t, b, g, row0, L, nkv, kt;
};
template <int KC, bool REUSE>
__device__ __forceinline__ FaTile fa_tile(const PrefillArgs& a, int tau) {
  FaTile x;
  const int BH = a.B * a.Hq;
  x.bh = tau % BH;
  x.t = a.nT - 1 - tau / BH;   // longest tiles first
  x.b = x.bh / a.Hq;
  x.g = a.head_kv[x.bh % a.Hq];
  x.row0 = x.t * kTile;
  x.L = min(a.N, x.row0 + kTile);
  x.kt = REUSE ? min(a.topk, x.L) : 0;
  x.nkv = REUSE ? (x.kt + KC - 1) / KC : (x.L + KC - 1) / KC;
  return x;
}

// n-th tile of this CTA: rounds of gridDim.x tiles in longest-first order,
// taken left to right in even rounds and right to left in odd ones, so the
// CTAs that get a round's longest tile get the next round's shortest.
__device__ __forceinline__ int fa_tau(int n) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return n * G + ((n & 1) ? G - 1 - c : c);
}

template <bool REUSE, bool LSE>
__global__ void __launch_bounds__(fa_threads<REUSE>(), 1)
    k_prefill_fa2(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const __grid_constant__ PrefillArgs a) {
  using SM = Fa2Smem<REUSE>;
  constexpr int kKC = SM::KC, kST = SM::ST;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int pipe, role;   // role: 0 softmax, 1 MMA, 2 producer, 3 Q loader
  if (warp < 8) { pipe = warp >> 2; role = 0; }
  else if (warp < 10) { pipe = warp - 8; role = 1; }
  else if (warp < fa_q_warp<REUSE>()) { pipe = (warp - 10) & 1; role = 2; }
  else { pipe = 0; role = 3; }

  unsigned char* ps = sm + (pipe ? SM::PIPE1 : SM::PIPE0);
  int32_t* s_pos = reinterpret_cast<int32_t*>(sm + SM::POS) + pipe * kST * kKC;
  // reuse: 1 if chunk stage s needs no causal mask
  int32_t* s_flag = reinterpret_cast<int32_t*>(sm + SM::POS) + 2 * kST * kKC + pipe * kST;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SM::BAR);
  uint64_t* q_full = bars + 2 * SM::NB;       // the tile's Q landed in shared memory
  uint64_t* q_ready = q_full + 1;             // ... and was copied into TMEM (both halves)
  // o_ready[m & 1]: tile m's output is staged where Q was (two barriers, so a
  // phase is reused only after the Q loader has waited for it: tile m + 2
  // needs the Q that is loaded after tile m's output left)
  uint64_t* o_ready = q_full + 2;
  uint64_t* bar = bars + pipe * SM::NB;
  uint64_t* kv_full = bar;                    // [kST]
  uint64_t* kv_free = bar + kST;              // [kST]
  uint64_t* s_full = bar + 2 * kST;           // scores of the current chunk
  uint64_t* s_free = s_full + 1;              // ... read by the softmax
  uint64_t* p_full = s_full + 2;              // P of the current chunk written
  uint64_t* pv_done = s_full + 3;             // its P V product completed
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + SM::TMEM);
  const uint32_t sQ = smem_u32(sm + SM::Q), sK0 = smem_u32(ps + SM::K0);
  const uint32_t sV0 = smem_u32(ps + SM::V0);
  const int total = a.B * a.Hq * a.nT;

  if (threadIdx.x < 2) {   // thread p initialises pipe p's barriers
    uint64_t* pb = bars + threadIdx.x * SM::NB;
    for (int s = 0; s < kST; ++s) {
      mbar_init(pb + s, REUSE ? 32 : 1);
      mbar_init(pb + kST + s, 1);
    }
    mbar_init(pb + 2 * kST, 1);         // s_full
    mbar_init(pb + 2 * kST + 1, 128);   // s_free
    mbar_init(pb + 2 * kST + 2, 128);   // p_full
    mbar_init(pb + 2 * kST + 3, 1);     // pv_done
    if (threadIdx.x == 0) {
      mbar_init(q_full, 1);
      mbar_init(q_ready, 256);
      mbar_init(o_ready, 256);
      mbar_init(o_ready + 1, 256);
    }
    fence_barrier_init();
  }
  if (warp == 8) tmem_alloc(s_tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const uint32_t tQ = tmem_base;
  const uint32_t tS = tmem_base + SM::T_PIPE + pipe * SM::T_PIPE_COLS + SM::T_S;
  const uint32_t tP = tS - SM::T_S + SM::T_P, tO = tS - SM::T_S + SM::T_O;

  if (role == 3) {
    // ------------------------------------------------ Q loads and output
    // stores through the Q staging area: Q(m) is loaded once the output of
    // tile m - 2 (staged there after Q(m - 1) went to TMEM) has been read out
    // by its TMA store; ragged tiles (past the sequence end) store their rows
    // themselves.
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmO);
      auto store_out = [&](int m) {   // output of this CTA's tile m
        if (!mbar_wait(o_ready + (m & 1), (m >> 1) & 1, a.err, 0x632)) return false;
        const FaTile x = fa_tile<kKC, REUSE>(a, fa_tau(m));
        if (x.row0 + kTile <= a.N) {
          tma_store_2d(&tmO, sm + SM::Q, 0, x.bh * a.N + x.row0);
          tma_store_2d(&tmO, sm + SM::Q + kHalf, 64, x.bh * a.N + x.row0);
          bulk_commit_group();
          bulk_wait_group_read0();   // the staging area may take the next Q
        }
        return true;
      };
      int n = 0, stored = 0;
      bool ok = true;
      for (int tau = fa_tau(0); ok && tau < total; tau = fa_tau(++n)) {
        if (n == 1) ok = mbar_wait(q_ready, 0, a.err, 0x630);
        if (n >= 2) {
          ok = store_out(n - 2);
          stored = n - 1;
        }
        if (!ok) break;
        const FaTile x = fa_tile<kKC, REUSE>(a, tau);
        mbar_arrive_expect_tx(q_full, kTileBytes);
        tma_load_2d(sm + SM::Q, &tmQ, q_full, 0, x.bh * a.N + x.row0);
        tma_load_2d(sm + SM::Q + kHalf, &tmQ, q_full, 64, x.bh * a.N + x.row0);
      }
      for (int m = stored; ok && fa_tau(m) < total; ++m) ok = store_out(m);
      bulk_wait_group0();   // every output store has landed
      if (n > 0) mbar_wait(q_full, (n - 1) & 1, a.err, 0x631);   // no copy left in flight
    }
  } else if (role == 2) {
    // ------------------------------------------------ producers
    if (!REUSE) {
      if (lane == 0) {   // one TMA producer per pipeline
        uint32_t c = 0;   // this pipe's chunks so far, over all tiles
        bool ok = true;
        int n = 0;
        for (int tau = fa_tau(0); ok && tau < total; tau = fa_tau(++n)) {
          const FaTile x = fa_tile<kKC, REUSE>(a, tau);
          const int np = (x.nkv - pipe + 1) / 2;
          const int kv_row_base = (x.b * a.Hkv + x.g) * a.N;
          for (int i = 0; i < np; ++i) {
            const uint32_t gi = c + i;
            const int s = gi % kST;
            if (!mbar_wait(kv_free + s, ((gi / kST) & 1) ^ 1, a.err, 0x601)) {
              ok = false;
              c = gi;
              break;
            }
            unsigned char* kd = ps + SM::K0 + s * SM::KV_BYTES;
            unsigned char* vd = ps + SM::V0 + s * SM::KV_BYTES;
            mbar_arrive_expect_tx(kv_full + s, 2 * SM::KV_BYTES);
            const int y = kv_row_base + (2 * i + pipe) * kKC;
            tma_load_2d(kd, &tmK, kv_full + s, 0, y);
            tma_load_2d(kd + SM::KHALF, &tmK, kv_full + s, 64, y);
            tma_load_2d(vd, &tmV, kv_full + s, 0, y);
            tma_load_2d(vd + SM::KHALF, &tmV, kv_full + s, 64, y);
          }
          if (ok) c += np;
        }
        // never leave with copies in flight: the last kST chunks issued
        for (uint32_t gi = c > kST ? c - kST : 0; gi < c; ++gi)
          mbar_wait(kv_full + (gi % kST), (gi / kST) & 1, a.err, 0x604);
      }
    } else {
      // kProd gather warps per pipeline take its chunks in turn (global chunk
      // gi of the pipe goes to warp gi % kProd), each with up to kDepth of its
      // chunks in flight: a chunk is released (kv_full) once its copies have
      // landed. Before waiting for a ring stage that is still busy, a warp
      // releases every chunk it has in flight, so the MMA issuer never waits
      // on copies held back behind that wait. Within a tile, positions are
      // read one chunk ahead.
      constexpr int kProd = 2;
      constexpr int kDepth = 2;
      const int prod = (warp - 10) >> 1;
      const int sub = lane >> 4, c16 = lane & 15;
      // this lane's swizzled 16-byte column in shared memory for rows
      // congruent to 2u + sub (mod 8)
      uint32_t sw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        sw[u] = (c16 >> 3) * SM::KHALF + sub * 128 + (((c16 & 7) ^ ((2 * u + sub) & 7)) << 4);
      auto release_all = [&](uint32_t from, uint32_t to) {   // own chunks from, from + kProd, ... < to
        cp_async_wait<0>();
        fence_proxy_async_smem();
        for (uint32_t c2 = from; c2 < to; c2 += kProd) mbar_arrive(kv_full + c2 % kST);
      };
      uint32_t c = 0;                                   // this pipe's chunks so far
      uint32_t issued = prod, released = prod;          // own chunks [released, issued) in flight
      bool ok = true;
      int n = 0;
      for (int tau = fa_tau(0); ok && tau < total; tau = fa_tau(++n)) {
        const FaTile x = fa_tile<kKC, REUSE>(a, tau);
        const int np = (x.nkv - pipe + 1) / 2;
        const int32_t* idx_row = a.idx + (static_cast<size_t>(x.bh) * a.nT + x.t) * a.topk;
        const int kv_row_base = (x.b * a.Hkv + x.g) * a.N;
        const __nv_bfloat16* kl = static_cast<const __nv_bfloat16*>(a.k) +
                                  static_cast<size_t>(kv_row_base) * 128 + c16 * 8;
        const __nv_bfloat16* vl = static_cast<const __nv_bfloat16*>(a.v) +
                                  static_cast<size_t>(kv_row_base) * 128 + c16 * 8;
        auto read_pos = [&](int i, int (&pos)[kKC / 32]) {
#pragma unroll
          for (int half = 0; half < kKC / 32; ++half) {
            const int e = (2 * i + pipe) * kKC + lane + 32 * half;
            pos[half] = e < x.kt ? __ldg(idx_row + e) : -1;
          }
        };
        // this warp's first chunk of the tile: global chunk c + i0 = prod (mod kProd)
        const int i0 = static_cast<int>((prod + kProd - c % kProd) % kProd);
        int p_first = 0;
        int nxt[kKC / 32];
        if (i0 < np) {
          p_first = __ldg(idx_row);
          if (p_first < 0 || p_first >= a.N) p_first = 0;
          read_pos(i0, nxt);
        }
        for (int i = i0; i < np; i += kProd) {
          const uint32_t gi = c + i;
          const int s = gi % kST, j = 2 * i + pipe;
          int pos[kKC / 32];
#pragma unroll
          for (int half = 0; half < kKC / 32; ++half) pos[half] = nxt[half];
          if (i + kProd < np) read_pos(i + kProd, nxt);
          const uint32_t par = ((gi / kST) & 1) ^ 1;
          int ready = lane == 0 ? mbar_test_wait(kv_free + s, par) : 0;
          if (!__shfl_sync(0xffffffffu, ready, 0)) {
            release_all(released, issued);
            released = issued;
            int okw = 1;
            if (lane == 0) okw = mbar_wait(kv_free + s, par, a.err, 0x605);
            if (!__shfl_sync(0xffffffffu, okw, 0)) {
              ok = false;
              break;
            }
          }
          const uint32_t kd = smem_u32(ps + SM::K0 + s * SM::KV_BYTES);
          const uint32_t vd = smem_u32(ps + SM::V0 + s * SM::KV_BYTES);
          // validate; padding slots (-1) re-read the tile's first saved row
          // and are masked later
          int src[kKC / 32], pmax = -1;
          bool all_valid = true;
#pragma unroll
          for (int half = 0; half < kKC / 32; ++half) {
            const int pt = lane + 32 * half;
            const int e = j * kKC + pt;
            int p = pos[half];
            if (p >= a.N || (e < x.kt && p < 0)) {
              report_error(a.err, KASCADE_ERR_BAD_INPUT, 0x602);
              p = -1;
            }
            s_pos[s * kKC + pt] = p;
            src[half] = p >= 0 ? p : p_first;
            all_valid = all_valid && p >= 0;
            pmax = max(pmax, p);
          }
          // a chunk of valid keys that all precede the tile's first row
          // needs no causal mask in any of its rows
          all_valid = __all_sync(0xffffffffu, all_valid);
          pmax = __reduce_max_sync(0xffffffffu, pmax);
          if (lane == 0) s_flag[s] = (all_valid && pmax <= x.row0) ? 1 : 0;
          // coalesced copies: a half-warp moves one 256-byte row (16 lanes x
          // 16 bytes), so each instruction fills two rows of K (or V) in full
#pragma unroll
          for (int rr = 0; rr < kKC / 2; ++rr) {
            const int prow = __shfl_sync(0xffffffffu, src[(2 * rr) >> 5], (2 * rr + sub) & 31);
            const uint32_t off = sw[rr & 3] + rr * 256;
            cp_async16_s(kd + off, kl + static_cast<size_t>(prow) * 128);
            cp_async16_s(vd + off, vl + static_cast<size_t>(prow) * 128);
          }
          cp_async_commit();
          issued = gi + kProd;
          if (issued - released >= kDepth * kProd) {   // the oldest own chunk in flight has landed
            cp_async_wait<kDepth - 1>();
            fence_proxy_async_smem();
            mbar_arrive(kv_full + released % kST);
            released += kProd;
          }
        }
        c += np;
      }
      // release what is still in flight (also after an error, so that no copy
      // outlives the kernel)
      release_all(released, issued);
    }
  } else if (role == 1) {
    // ------------------------------------------------ MMA issuer (the whole
    // warp runs the loop; one elected lane issues each MMA)
    constexpr uint32_t idq = idesc_bf16_f32(128, kKC, 0, 0);
    constexpr uint32_t idv = idesc_bf16_f32(128, 128, 0, 1);
    uint32_t c = 0;   // this pipe's chunks so far, over all tiles
    // S = Q K^T of global chunk gi (A = Q from TMEM) once the softmax has read
    // the previous scores
    auto issue_s = [&](uint32_t gi) {
      const int s = gi % kST;
      if (!mbar_wait(kv_full + s, (gi / kST) & 1, a.err, 0x613)) return false;
      if (gi > 0 && !mbar_wait(s_free, (gi - 1) & 1, a.err, 0x614)) return false;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc_mma_ts(tS, tQ + kk * 8, kmajor_desc(sK0 + s * SM::KV_BYTES, kk, SM::KHALF), idq,
                  kk > 0 ? 1u : 0u);
      tc_commit(s_full);
      return true;
    };
    // O += P V with P (A operand) from its own TMEM columns; the tile's first
    // product overwrites O
    auto issue_pv = [&](uint32_t gi, bool first) {
      const int s = gi % kST;
      if (!mbar_wait(p_full, gi & 1, a.err, 0x612)) return false;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kKC / 16; ++kk)
        tc_mma_ts(tO, tP + kk * 8, vmn_desc(sV0 + s * SM::KV_BYTES, kk, SM::KHALF), idv,
                  (!first || kk > 0) ? 1u : 0u);
      tc_commit(pv_done);
      tc_commit(kv_free + s);
      return true;
    };
    bool ok = true;
    int n = 0;
    for (int tau = fa_tau(0); ok && tau < total; tau = fa_tau(++n)) {
      const FaTile x = fa_tile<kKC, REUSE>(a, tau);
      const int np = (x.nkv - pipe + 1) / 2;
      ok = mbar_wait(q_ready, n & 1, a.err, 0x611);   // this tile's Q is in TMEM
      if (!ok) break;
      tc_fence_after();
      if (np > 0) ok = issue_s(c);
      for (int i = 0; ok && i < np; ++i) {
        if (i + 1 < np) ok = issue_s(c + i + 1);
        if (ok) ok = issue_pv(c + i, i == 0);
      }
      c += np;
    }
  } else {
    // ------------------------------------------------ softmax warpgroups
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    // at the end of a tile each pipe's (then idle) P columns carry its (m, l)
    // to the other pipe; pipe p merges output dims [64 p, 64 p + 64)
    const uint32_t tXchOwn = tP, tXchOther = tmem_base + SM::T_PIPE +
                                             (1 - pipe) * SM::T_PIPE_COLS + SM::T_P;
    const uint32_t tOa = tmem_base + SM::T_PIPE + SM::T_O;                      // pipe 0's O
    const uint32_t tOb = tmem_base + SM::T_PIPE + SM::T_PIPE_COLS + SM::T_O;    // pipe 1's O
    bool ok = true;
    // the Q tile (128-byte-swizzled halves in shared memory) into TMEM columns
    // [0, 64) as bf16 pairs, one row per thread
    // pipe p copies dims [64p, 64p + 64) of the Q tile (its 128-byte-swizzled
    // half in shared memory) into TMEM columns [32p, 32p + 32) as bf16 pairs,
    // one row per thread; later it stages its half of the output there
    auto copy_q = [&](int n) {
      if (ok) ok = mbar_wait(q_full, n & 1, a.err, 0x620);
      uint32_t qv[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t addr = sQ + pipe * kHalf + r * 128 + ((c ^ (r & 7)) << 4);
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(qv[c * 4]), "=r"(qv[c * 4 + 1]), "=r"(qv[c * 4 + 2]),
                       "=r"(qv[c * 4 + 3])
                     : "r"(addr));
      }
      tmem_st32(tQ + pipe * 32 + lane_base, qv);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_ready);
    };
    if (fa_tau(0) < total) copy_q(0);
    uint32_t c = 0;   // this pipe's chunks so far, over all tiles
    int n = 0;
    // Every softmax thread walks every tile (also after an error, skipping the
    // waits), so the two named barriers per tile always pair up.
    for (int tau = fa_tau(0); tau < total; tau = fa_tau(++n)) {
      const FaTile x = fa_tile<kKC, REUSE>(a, tau);
      const int np = (x.nkv - pipe + 1) / 2;
      const int row = x.row0 + r;
      float m_used = kNegInfP, l = 0.f;
      for (int i = 0; ok && i < np; ++i) {
        const uint32_t gi = c + i;
        const int s = gi % kST, j = 2 * i + pipe;
        ok = mbar_wait(s_full, gi & 1, a.err, 0x621);
        if (!ok) break;
        tc_fence_after();
        float xv[kKC];
#pragma unroll
        for (int cc = 0; cc < kKC / 32; ++cc) {
          uint32_t v[32];
          tmem_ld32(tS + cc * 32 + lane_base, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) xv[cc * 32 + e] = __uint_as_float(v[e]);
        }
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(s_free);   // the score buffer may take the next S now
        const bool need_mask = REUSE ? (s_flag[s] == 0) : (j * kKC + kKC - 1 > x.row0);
        if (need_mask) {
#pragma unroll
          for (int cc = 0; cc < kKC; ++cc) {
            const int kp = REUSE ? s_pos[s * kKC + cc] : j * kKC + cc;
            if (!(kp >= 0 && kp <= row)) xv[cc] = kNegInfP;
          }
        }
        // row maximum: eight chains of three-input maxima
        float mx[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) mx[cc] = fmaxf(xv[2 * cc], xv[2 * cc + 1]);
#pragma unroll
        for (int cc = 8; cc < kKC / 2; ++cc) mx[cc & 7] = fmax3(mx[cc & 7], xv[2 * cc], xv[2 * cc + 1]);
        float tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        tmax *= a.scale_log2;
        float alpha = 1.f;
        bool resc = false;
        if (tmax > m_used + kRescaleLog2) {
          if (i > 0) {
            alpha = ex2_approx(m_used - tmax);
            resc = true;
          }
          l *= alpha;
          m_used = tmax;
        }
        const float mu = (m_used == kNegInfP) ? 0.f : m_used;
        // exponents and row sums on packed pairs (one FMA / add per two scores)
        const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2), nmu2 = f2_pack(-mu, -mu);
        uint32_t pk[kKC / 2];
        uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int cc = 0; cc < kKC / 2; ++cc) {
          float y0, y1;
          f2_unpack(f2_fma(f2_pack(xv[2 * cc], xv[2 * cc + 1]), sc2, nmu2), y0, y1);
          const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
          ls2[cc & 3] = f2_add(ls2[cc & 3], f2_pack(p0, p1));
          pk[cc] = pack_bf16(p0, p1);
        }
        {
          float s0, s1;
          f2_unpack(f2_add(f2_add(ls2[0], ls2[1]), f2_add(ls2[2], ls2[3])), s0, s1);
          l += s0 + s1;
        }
        // the P columns and O are free once the previous P V product has landed
        if (gi > 0) {
          ok = mbar_wait(pv_done, (gi - 1) & 1, a.err, 0x622);
          if (!ok) break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32 + lane_base, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + cc * 32 + lane_base, o);
          }
        }
        tmem_store_p<kKC>(tP + lane_base, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full);
      }
      // wait for this pipe's last P V of the tile (it also covers every S)
      if (ok && np > 0) ok = mbar_wait(pv_done, (c + np - 1) & 1, a.err, 0x623);
      c += np;
      tc_fence_after();
      {
        uint32_t xw[16];
        xw[0] = __float_as_uint(np > 0 ? m_used : kNegInfP);
        xw[1] = __float_as_uint(np > 0 ? l : 0.f);
#pragma unroll
        for (int e = 2; e < 16; ++e) xw[e] = 0u;
        tmem_st16(tXchOwn + lane_base, xw);
        tmem_wait_st();
      }
      tc_fence_before();
      asm volatile("bar.sync 1, 256;" ::: "memory");   // both pipes done with the tile
      tc_fence_after();
      // the next tile's Q into TMEM first, so its scores overlap this merge
      if (fa_tau(n + 1) < total) copy_q(n + 1);
      {
        uint32_t xr[32];
        tmem_ld32(tXchOther + lane_base, xr);
        tmem_wait_ld();
        const float mo = __uint_as_float(xr[0]), lo = __uint_as_float(xr[1]);
        const float mine_m = np > 0 ? m_used : kNegInfP, mine_l = np > 0 ? l : 0.f;
        const float m0 = pipe == 0 ? mine_m : mo, l0 = pipe == 0 ? mine_l : lo;
        const float m1 = pipe == 0 ? mo : mine_m, l1 = pipe == 0 ? lo : mine_l;
        const float M = fmaxf(m0, m1);
        const float a0 = (m0 == kNegInfP) ? 0.f : ex2_approx(m0 - M);
        const float a1 = (m1 == kNegInfP) ? 0.f : ex2_approx(m1 - M);
        const float lt = a0 * l0 + a1 * l1;
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        __nv_bfloat16* orow =
            static_cast<__nv_bfloat16*>(a.out) + (static_cast<size_t>(x.bh) * a.N + row) * kTile;
        const bool full = x.row0 + kTile <= a.N;   // whole tile inside the sequence: TMA store
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int cc = 2 * pipe + h2;   // 32-dim block of the output
          uint32_t o0[32], o1[32];
          tmem_ld32(tOa + cc * 32 + lane_base, o0);
          tmem_ld32(tOb + cc * 32 + lane_base, o1);
          tmem_wait_ld();
          uint32_t ob[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float y0 = a0 * __uint_as_float(o0[2 * e]);
            float y1 = a0 * __uint_as_float(o0[2 * e + 1]);
            if (a1 != 0.f) {
              y0 += a1 * __uint_as_float(o1[2 * e]);
              y1 += a1 * __uint_as_float(o1[2 * e + 1]);
            }
            ob[e] = ok ? pack_bf16(y0 * inv, y1 * inv) : 0u;
          }
          if (full) {
            // into this pipe's (128-byte-swizzled) half of the staging area
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t addr = sQ + pipe * kHalf + r * 128 + (((h2 * 4 + q) ^ (r & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(ob[4 * q]),
                           "r"(ob[4 * q + 1]), "r"(ob[4 * q + 2]), "r"(ob[4 * q + 3])
                           : "memory");
            }
          } else if (row < a.N) {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(ob[4 * q], ob[4 * q + 1], ob[4 * q + 2], ob[4 * q + 3]);
          }
        }
        if (LSE && pipe == 0 && row < a.N)
          a.lse[static_cast<size_t>(x.bh) * a.N + row] = lt > 0.f ? M + __log2f(lt) : kNegInfP;
        fence_proxy_async_smem();   // staged rows visible to the TMA store
        mbar_arrive(o_ready + (n & 1));
      }
      tc_fence_before();
      asm volatile("bar.sync 1, 256;" ::: "memory");   // both O and P columns free again
      tc_fence_after();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------------
// Reuse prefill over GQA-pooled sets: the query heads of one KV head read the
// same saved rows, so a CTA takes two of them (one per pipeline) for one tile
// and both pipelines consume every gathered chunk. Per FLOP this halves the
// gathers of the per-head kernel above, whose pipelines split the chunks of
// one head. Q stays in shared memory (two 128-row tiles) and is the A operand
// of S = Q K^T; each pipeline keeps its own S, P and O columns in TMEM and
// writes its own head's rows, so there is no merge. One kPairST-deep ring of
// K/V chunks is filled by four gather warps (chunks j = w, w + 4, ...) and a
// stage is freed once both pipelines' P V products that read it completed.
// Warps: 0-3 softmax of pipe 0, 4-7 softmax of pipe 1, 8/9 MMA of pipe 0/1,
// 10-13 gathers.
constexpr int kPairThreads = 448;
constexpr int kPairST = 5;

struct PairSmem {
  static constexpr int KC = 64, ST = kPairST;
  static constexpr int KHALF = KC * 128;              // one 64-dim half of a K (or V) chunk
  static constexpr int KV_BYTES = 2 * KHALF;          // a K (or V) chunk
  static constexpr int STAGE = 2 * KV_BYTES;          // K, then V
  static constexpr int Q = 0;                         // two 128-row Q tiles
  static constexpr int RING = 2 * kTileBytes;
  static constexpr int POS = RING + ST * STAGE;       // int32 positions [ST][KC], flags [ST]
  static constexpr int POS_BYTES = ST * (KC + 1) * 4;
  static constexpr int NB = 2 * ST + 8 + 1;           // kv_full, kv_free, 4 per pipe, q_full
  static constexpr int BAR = (POS + POS_BYTES + 7) & ~7;
  static constexpr int TMEM = BAR + NB * 8;
  static constexpr int BYTES = TMEM + 8;
  static constexpr size_t SMEM = BYTES + 1024;        // + slack for 1024-byte alignment
  static_assert(SMEM <= 232448, "two Q tiles and the ring must fit in shared memory");
  static_assert(RING % 1024 == 0 && STAGE % 1024 == 0, "swizzled tiles are 1024-byte aligned");
  // TMEM columns of pipeline p at 224 p: S (KC fp32), P (KC / 2 bf16 pairs), O (128)
  static constexpr int T_PIPE_COLS = 224, T_S = 0, T_P = 64, T_O = 96;
  static_assert(2 * T_PIPE_COLS <= 512, "two pipelines in TMEM");
};

__global__ void __launch_bounds__(kPairThreads, 1)
    k_prefill_pair(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ PrefillArgs a) {
  using SM = PairSmem;
  constexpr int kKC = SM::KC, kST = SM::ST;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int pipe, role;   // role: 0 softmax, 1 MMA, 2 gather
  if (warp < 8) { pipe = warp >> 2; role = 0; }
  else if (warp < 10) { pipe = warp - 8; role = 1; }
  else { pipe = 0; role = 2; }

  int32_t* s_pos = reinterpret_cast<int32_t*>(sm + SM::POS);   // [kST][kKC]
  int32_t* s_flag = s_pos + kST * kKC;                          // [kST]: 1 = no causal mask
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SM::BAR);
  uint64_t* kv_full = bars;                   // [kST] chunk landed (32 lanes of its gather warp)
  uint64_t* kv_free = bars + kST;             // [kST] both pipelines' P V read it
  uint64_t* pb = bars + 2 * kST + 4 * pipe;
  uint64_t* s_full = pb;                      // scores of the current chunk
  uint64_t* s_free = pb + 1;                  // ... read by the softmax
  uint64_t* p_full = pb + 2;                  // P of the current chunk written
  uint64_t* pv_done = pb + 3;                 // its P V product completed
  uint64_t* q_full = bars + 2 * kST + 8;      // both Q tiles landed
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + SM::TMEM);

  const int GP = a.G >> 1;                    // head pairs per KV head
  const int units = a.B * a.Hkv * GP;
  const int u = static_cast<int>(blockIdx.x) % units;
  const int t = a.nT - 1 - static_cast<int>(blockIdx.x) / units;   // longest tiles first
  const int b = u / (a.Hkv * GP), g = (u / GP) % a.Hkv, hp = u % GP;
  const int row0 = t * kTile;
  const int L = min(a.N, row0 + kTile);
  const int kt = min(a.topk, L);
  const int nkv = (kt + kKC - 1) / kKC;
  const int32_t* idx_row = a.idx + ((static_cast<size_t>(b) * a.Hkv + g) * a.nT + t) * a.topk;
  const int kv_row_base = (b * a.Hkv + g) * a.N;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kST; ++s) {
      mbar_init(kv_full + s, 32);
      mbar_init(kv_free + s, 2);
    }
    for (int p = 0; p < 2; ++p) {
      uint64_t* q = bars + 2 * kST + 4 * p;
      mbar_init(q, 1);         // s_full
      mbar_init(q + 1, 128);   // s_free
      mbar_init(q + 2, 128);   // p_full
      mbar_init(q + 3, 1);     // pv_done
    }
    mbar_init(q_full, 1);
    fence_barrier_init();
  }
  if (warp == 8) tmem_alloc(s_tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const uint32_t tS = tmem_base + pipe * SM::T_PIPE_COLS + SM::T_S;
  const uint32_t tP = tS - SM::T_S + SM::T_P, tO = tS - SM::T_S + SM::T_O;

  if (role == 2) {
    // ------------------------------------------------ gathers
    if (warp == 10 && lane == 0) {
      prefetch_tmap(&tmQ);
      mbar_arrive_expect_tx(q_full, 2 * kTileBytes);
      for (int p = 0; p < 2; ++p) {
        const int y = (b * a.Hq + a.heads[g * a.G + 2 * hp + p]) * a.N + row0;
        tma_load_2d(sm + SM::Q + p * kTileBytes, &tmQ, q_full, 0, y);
        tma_load_2d(sm + SM::Q + p * kTileBytes + kHalf, &tmQ, q_full, 64, y);
      }
    }
    // Warp 10 + w gathers chunks j = w, w + 4, ... with up to kDepth of them
    // in flight; a chunk is released (kv_full) once its copies have landed.
    // Before waiting for a ring stage that is still busy a warp releases every
    // chunk it has in flight, so no pipeline waits on copies held back behind
    // that wait. Positions are read one chunk ahead.
    constexpr int kProd = 4, kDepth = 2;
    const int w0 = warp - 10;
    int p_first = __ldg(idx_row);
    if (p_first < 0 || p_first >= a.N) p_first = 0;
    const int sub = lane >> 4, c16 = lane & 15;
    const __nv_bfloat16* kl = static_cast<const __nv_bfloat16*>(a.k) +
                              static_cast<size_t>(kv_row_base) * 128 + c16 * 8;
    const __nv_bfloat16* vl = static_cast<const __nv_bfloat16*>(a.v) +
                              static_cast<size_t>(kv_row_base) * 128 + c16 * 8;
    uint32_t sw[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      sw[q] = (c16 >> 3) * SM::KHALF + sub * 128 + (((c16 & 7) ^ ((2 * q + sub) & 7)) << 4);
    auto read_pos = [&](int j, int (&pos)[kKC / 32]) {
#pragma unroll
      for (int half = 0; half < kKC / 32; ++half) {
        const int e = j * kKC + lane + 32 * half;
        pos[half] = e < kt ? __ldg(idx_row + e) : -1;
      }
    };
    auto release_all = [&](int from, int to) {   // own chunks from, from + kProd, ... < to
      cp_async_wait<0>();
      fence_proxy_async_smem();
      for (int c = from; c < to; c += kProd) mbar_arrive(kv_full + c % kST);
    };
    int nxt[kKC / 32];
    if (w0 < nkv) read_pos(w0, nxt);
    int issued = w0, released = w0;   // own chunks [released, issued) are in flight
    for (int j = w0; j < nkv; j += kProd) {
      const int s = j % kST;
      int pos[kKC / 32];
#pragma unroll
      for (int half = 0; half < kKC / 32; ++half) pos[half] = nxt[half];
      if (j + kProd < nkv) read_pos(j + kProd, nxt);
      const uint32_t par = ((j / kST) & 1) ^ 1;
      int ready = lane == 0 ? mbar_test_wait(kv_free + s, par) : 0;
      if (!__shfl_sync(0xffffffffu, ready, 0)) {
        release_all(released, issued);
        released = issued;
        int okw = 1;
        if (lane == 0) okw = mbar_wait(kv_free + s, par, a.err, 0x6a5);
        if (!__shfl_sync(0xffffffffu, okw, 0)) break;
      }
      const uint32_t kd = smem_u32(sm + SM::RING + s * SM::STAGE), vd = kd + SM::KV_BYTES;
      // validate; padding slots (-1) re-read the tile's first saved row and
      // are masked later
      int src[kKC / 32], pmax = -1;
      bool all_valid = true;
#pragma unroll
      for (int half = 0; half < kKC / 32; ++half) {
        const int pt = lane + 32 * half;
        const int e = j * kKC + pt;
        int p = pos[half];
        if (p >= a.N || (e < kt && p < 0)) {
          report_error(a.err, KASCADE_ERR_BAD_INPUT, 0x6a2);
          p = -1;
        }
        s_pos[s * kKC + pt] = p;
        src[half] = p >= 0 ? p : p_first;
        all_valid = all_valid && p >= 0;
        pmax = max(pmax, p);
      }
      // a chunk of valid keys that all precede the tile's first row needs no
      // causal mask in any of its rows
      all_valid = __all_sync(0xffffffffu, all_valid);
      pmax = __reduce_max_sync(0xffffffffu, pmax);
      if (lane == 0) s_flag[s] = (all_valid && pmax <= row0) ? 1 : 0;
      // coalesced copies: a half-warp moves one 256-byte row (16 lanes x 16
      // bytes), so each instruction fills two rows of K (or V) in full
#pragma unroll
      for (int rr = 0; rr < kKC / 2; ++rr) {
        const int prow = __shfl_sync(0xffffffffu, src[(2 * rr) >> 5], (2 * rr + sub) & 31);
        const uint32_t off = sw[rr & 3] + rr * 256;
        cp_async16_s(kd + off, kl + static_cast<size_t>(prow) * 128);
        cp_async16_s(vd + off, vl + static_cast<size_t>(prow) * 128);
      }
      cp_async_commit();
      issued = j + kProd;
      if (issued - released >= kDepth * kProd) {   // the oldest own chunk in flight has landed
        cp_async_wait<kDepth - 1>();
        fence_proxy_async_smem();
        mbar_arrive(kv_full + released % kST);
        released += kProd;
      }
    }
    // release what is still in flight (also after an error, so that no copy
    // outlives the kernel)
    release_all(released, issued);
    if (warp == 10 && lane == 0) mbar_wait(q_full, 0, a.err, 0x6a3);   // no copies left in flight
  } else if (role == 1) {
    // ------------------------------------------------ MMA issuer of pipe p
    constexpr uint32_t idq = idesc_bf16_f32(128, kKC, 0, 0);
    constexpr uint32_t idv = idesc_bf16_f32(128, 128, 0, 1);
    const uint32_t sQp = smem_u32(sm + SM::Q + pipe * kTileBytes);
    const uint32_t sRing = smem_u32(sm + SM::RING);
    bool ok = mbar_wait(q_full, 0, a.err, 0x6b1);
    // S = Q K^T of chunk i once the softmax has read S(i-1)
    auto issue_s = [&](int i) {
      const int s = i % kST;
      if (!mbar_wait(kv_full + s, (i / kST) & 1, a.err, 0x6b3)) return false;
      if (i > 0 && !mbar_wait(s_free, (i - 1) & 1, a.err, 0x6b4)) return false;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc_mma(tS, kmajor_desc(sQp, kk), kmajor_desc(sRing + s * SM::STAGE, kk, SM::KHALF), idq,
               kk > 0 ? 1u : 0u);
      tc_commit(s_full);
      return true;
    };
    // O += P V with P (A operand) from TMEM; the stage is freed for both pipes
    auto issue_pv = [&](int i) {
      const int s = i % kST;
      if (!mbar_wait(p_full, i & 1, a.err, 0x6b2)) return false;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kKC / 16; ++kk)
        tc_mma_ts(tO, tP + kk * 8, vmn_desc(sRing + s * SM::STAGE + SM::KV_BYTES, kk, SM::KHALF),
                  idv, (i > 0 || kk > 0) ? 1u : 0u);
      tc_commit(pv_done);
      tc_commit(kv_free + s);
      return true;
    };
    if (ok) tc_fence_after();
    if (ok && nkv > 0) ok = issue_s(0);
    for (int i = 0; ok && i < nkv; ++i) {
      if (i + 1 < nkv) ok = issue_s(i + 1);
      if (ok) ok = issue_pv(i);
    }
  } else {
    // ------------------------------------------------ softmax warpgroup of pipe p
    const int r = (warp & 3) * 32 + lane;
    const int row = row0 + r;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    float m_used = kNegInfP, l = 0.f;
    for (int i = 0; ok && i < nkv; ++i) {
      const int s = i % kST;
      ok = mbar_wait(s_full, i & 1, a.err, 0x6c1);
      if (!ok) break;
      tc_fence_after();
      float x[kKC];
#pragma unroll
      for (int c = 0; c < kKC / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tS + c * 32 + lane_base, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(v[e]);
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(s_free);   // the score columns may take S(i+1) now
      if (s_flag[s] == 0) {
#pragma unroll
        for (int c = 0; c < kKC; ++c) {
          const int kp = s_pos[s * kKC + c];
          if (!(kp >= 0 && kp <= row)) x[c] = kNegInfP;
        }
      }
      float mx[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) mx[c] = fmaxf(x[2 * c], x[2 * c + 1]);
#pragma unroll
      for (int c = 8; c < kKC / 2; ++c) mx[c & 7] = fmax3(mx[c & 7], x[2 * c], x[2 * c + 1]);
      float tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      tmax *= a.scale_log2;
      float alpha = 1.f;
      bool resc = false;
      if (tmax > m_used + kRescaleLog2) {
        if (i > 0) {
          alpha = ex2_approx(m_used - tmax);
          resc = true;
        }
        l *= alpha;
        m_used = tmax;
      }
      const float mu = (m_used == kNegInfP) ? 0.f : m_used;
      const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2), nmu2 = f2_pack(-mu, -mu);
      uint32_t pk[kKC / 2];
      uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int c = 0; c < kKC / 2; ++c) {
        float y0, y1;
        f2_unpack(f2_fma(f2_pack(x[2 * c], x[2 * c + 1]), sc2, nmu2), y0, y1);
        const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
        ls2[c & 3] = f2_add(ls2[c & 3], f2_pack(p0, p1));
        pk[c] = pack_bf16(p0, p1);
      }
      {
        float s0, s1;
        f2_unpack(f2_add(f2_add(ls2[0], ls2[1]), f2_add(ls2[2], ls2[3])), s0, s1);
        l += s0 + s1;
      }
      // the P columns and O are free once the previous P V product has landed
      if (i > 0) {
        ok = mbar_wait(pv_done, (i - 1) & 1, a.err, 0x6c2);
        if (!ok) break;
      }
      tc_fence_after();
      if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32 + lane_base, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + c * 32 + lane_base, o);
        }
      }
      tmem_store_p<kKC>(tP + lane_base, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok && nkv > 0) ok = mbar_wait(pv_done, (nkv - 1) & 1, a.err, 0x6c3);
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int hq = a.heads[g * a.G + 2 * hp + pipe];
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                          ((static_cast<size_t>(b) * a.Hq + hq) * a.N + row) * kTile;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      tmem_ld32(tO + c * 32 + lane_base, o);
      tmem_wait_ld();
      uint32_t ob[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        ob[e] = ok ? pack_bf16(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv)
                   : 0u;
      if (row < a.N) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(ob[4 * q], ob[4 * q + 1], ob[4 * q + 2], ob[4 * q + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------------
// Anchor pass 2: tile weights from S^T = K_j Q_t^T (TMEM lane = key).
// Persistent: one CTA per SM takes the (sequence, query head, 128-row) tiles
// in the same snake order as the attention kernel. Warp 0 loads each tile's
// Q (two buffers, so the next tile's Q and row LSEs land while the current
// tile is computed) and streams the key tiles 0..t through a kWtKS-deep TMA
// ring; warp 1 issues S^T(j) into TMEM score buffer kc % kWtSB (kc counts key
// tiles over all tiles of the CTA); kWtGroups epilogue warpgroups (warps 4-7,
// 8-11, ...) take the key tiles in turn (key tile kc goes to group
// kc % kWtGroups), each thread owning one key of the tile: it sums
// 2^(s*sigma*log2e - lse2) over the tile's query rows i >= key, with no
// cross-lane reduction.
// ------------------------------------------------------------------------
constexpr int kWtKS = 4;   // key-tile ring stages
constexpr int kWtSB = 4;   // TMEM score buffers (128 columns each)
struct WtSmem {
  static constexpr int Q = 0;                          // Q[2]
  static constexpr int K0 = Q + 2 * kTileBytes;        // K[kWtKS]
  static constexpr int LSE = K0 + kWtKS * kTileBytes;  // float [2][128], negated
  // q_full[2], q_free[2], k_full[KS], k_free[KS], s_full[SB], s_free[SB]
  static constexpr int BAR = LSE + 2 * kTile * 4;
  static constexpr int TMEM = BAR + (4 + 2 * kWtKS + 2 * kWtSB) * 8;
  static constexpr int BYTES = TMEM + 8;
};
constexpr size_t kWtSmemBytes = WtSmem::BYTES + 1024;
static_assert(kWtSmemBytes <= 232448, "weights kernel shared memory");

__global__ void __launch_bounds__(kWtThreads, 1)
    k_prefill_weights(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK, const __grid_constant__ PrefillArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* s_lse = reinterpret_cast<float*>(sm + WtSmem::LSE);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + WtSmem::BAR);
  uint64_t* q_full = bar;                          // [2] Q landed (tx) + LSE written (32 lanes)
  uint64_t* q_free = bar + 2;                      // [2] the tile's MMAs and epilogues are done
  uint64_t* k_full = bar + 4;                      // [kWtKS]
  uint64_t* k_free = k_full + kWtKS;               // [kWtKS]
  uint64_t* s_full = k_free + kWtKS;               // [kWtSB]
  uint64_t* s_free = s_full + kWtSB;               // [kWtSB]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + WtSmem::TMEM);
  const uint32_t sQ = smem_u32(sm + WtSmem::Q), sK0 = smem_u32(sm + WtSmem::K0);
  const int total = a.B * a.Hq * a.nT;
  const int BH = a.B * a.Hq;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t per_bh = static_cast<size_t>(64) * (a.nT - 1) * a.nT + a.N;

  if (threadIdx.x == 0) {
    for (int q = 0; q < 2; ++q) {
      mbar_init(q_full + q, 33);
      mbar_init(q_free + q, 1 + 128 * kWtGroups);
    }
    for (int s = 0; s < kWtKS; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_free + s, 1);
    }
    for (int s = 0; s < kWtSB; ++s) {
      mbar_init(s_full + s, 1);
      mbar_init(s_free + s, 128);
    }
    fence_barrier_init();
  }
  if (warp == 2) tmem_alloc(s_tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0) {
    // ------------------------------------------------ loads (whole warp)
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
    }
    uint32_t kc = 0;   // key tiles issued over all tiles of this CTA
    int n = 0, nq = 0;
    bool ok = true;
    for (int tau = fa_tau(0); ok && tau < total; tau = fa_tau(++n)) {
      const int bh = tau % BH, t = a.nT - 1 - tau / BH;
      const int b = bh / a.Hq, g = a.head_kv[bh % a.Hq];
      const int row0 = t * kTile;
      const int L = min(a.N, row0 + kTile);
      const int nkv = (L + kTile - 1) / kTile;
      const int buf = n & 1;
      // buffer buf is free once tile n - 2 is done with it
      int okw = 1;
      if (n >= 2 && lane == 0) okw = mbar_wait(q_free + buf, ((n >> 1) - 1) & 1, a.err, 0x704);
      if (!__shfl_sync(0xffffffffu, okw, 0)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full + buf, kTileBytes);
        tma_load_2d(sm + WtSmem::Q + buf * kTileBytes, &tmQ, q_full + buf, 0, bh * a.N + row0);
        tma_load_2d(sm + WtSmem::Q + buf * kTileBytes + kHalf, &tmQ, q_full + buf, 64,
                    bh * a.N + row0);
      }
      // the tile's row LSEs, stored negated (the epilogue's FMA adds them)
#pragma unroll
      for (int u = 0; u < kTile / 32; ++u) {
        const int rr = u * 32 + lane, i = row0 + rr;
        s_lse[buf * kTile + rr] =
            i < a.N ? -a.lse[static_cast<size_t>(bh) * a.N + i] : -CUDART_INF_F;
      }
      mbar_arrive(q_full + buf);
      nq = n + 1;
      if (lane == 0) {
        const int kv_row_base = (b * a.Hkv + g) * a.N;
        for (int j = 0; j < nkv; ++j) {
          const uint32_t gk = kc + j;
          const int s = gk % kWtKS;
          if (!mbar_wait(k_free + s, ((gk / kWtKS) & 1) ^ 1, a.err, 0x701)) {
            okw = 0;
            kc = gk;
            break;
          }
          unsigned char* kd = sm + WtSmem::K0 + s * kTileBytes;
          mbar_arrive_expect_tx(k_full + s, kTileBytes);
          tma_load_2d(kd, &tmK, k_full + s, 0, kv_row_base + j * kTile);
          tma_load_2d(kd + kHalf, &tmK, k_full + s, 64, kv_row_base + j * kTile);
        }
        if (okw) kc += nkv;
      }
      kc = __shfl_sync(0xffffffffu, kc, 0);
      if (!__shfl_sync(0xffffffffu, okw, 0)) ok = false;
    }
    // never leave with copies in flight
    if (lane == 0) {
      for (int m = nq > 2 ? nq - 2 : 0; m < nq; ++m)
        mbar_wait(q_full + (m & 1), (m >> 1) & 1, a.err, 0x702);
      for (uint32_t gk = kc > kWtKS ? kc - kWtKS : 0; gk < kc; ++gk)
        mbar_wait(k_full + (gk % kWtKS), (gk / kWtKS) & 1, a.err, 0x703);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (the whole
    // warp runs the loop; one elected lane issues each MMA)
    constexpr uint32_t id = idesc_bf16_f32(128, 128, 0, 0);
    uint32_t kc = 0;
    int n = 0;
    bool ok = true;
    for (int tau = fa_tau(0); ok && tau < total; tau = fa_tau(++n)) {
      const int t = a.nT - 1 - tau / BH;
      const int nkv = (min(a.N, t * kTile + kTile) + kTile - 1) / kTile;
      const int buf = n & 1;
      ok = mbar_wait(q_full + buf, (n >> 1) & 1, a.err, 0x711);
      const uint32_t sQb = sQ + buf * kTileBytes;
      for (int j = 0; ok && j < nkv; ++j) {
        const uint32_t gk = kc + j;
        const int s = gk % kWtKS, sb = gk % kWtSB;
        ok = mbar_wait(k_full + s, (gk / kWtKS) & 1, a.err, 0x712) &&
             mbar_wait(s_free + sb, ((gk / kWtSB) & 1) ^ 1, a.err, 0x713);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma(tmem + sb * 128, kmajor_desc(sK0 + s * kTileBytes, kk), kmajor_desc(sQb, kk), id,
                 kk > 0 ? 1u : 0u);
        tc_commit(s_full + sb);
        tc_commit(k_free + s);
      }
      if (ok) tc_commit(q_free + buf);   // this tile's Q buffer, once its MMAs complete
      kc += nkv;
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ epilogue groups
    const int grp = (warp - 4) >> 2;
    const int r = (warp & 3) * 32 + lane;   // key lane within the key tile
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
    uint32_t kc = 0;
    int n = 0;
    bool ok = true;
    for (int tau = fa_tau(0); tau < total; tau = fa_tau(++n)) {
      const int bh = tau % BH, t = a.nT - 1 - tau / BH;
      const int row0 = t * kTile;
      const int L = min(a.N, row0 + kTile);
      const int nkv = (L + kTile - 1) / kTile;
      const int buf = n & 1;
      // this group's key tiles of the tile: global key tile kc + j = grp (mod kWtGroups)
      const int j0 = static_cast<int>((grp + kWtGroups - kc % kWtGroups) % kWtGroups);
      // every thread waits for the tile's Q and LSEs, even with no key tile of
      // its own, so its arrival on q_free below belongs to this use of buf
      if (ok) ok = mbar_wait(q_full + buf, (n >> 1) & 1, a.err, 0x722);
      float* wrow = a.w + static_cast<size_t>(bh) * per_bh + static_cast<size_t>(64) * t * (t + 1);
      const uint64_t* lse2 = reinterpret_cast<const uint64_t*>(s_lse + buf * kTile);
      for (int j = j0; ok && j < nkv; j += kWtGroups) {
        const uint32_t gk = kc + j;
        const int sb = gk % kWtSB;
        if (!mbar_wait(s_full + sb, (gk / kWtSB) & 1, a.err, 0x721)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int kj = j * kTile + r;
        const uint32_t ts = tmem + sb * 128 + lane_base;
        // only the diagonal key tile (j == t) needs the causal mask i >= key;
        // exponents and sums on packed pairs of query columns, 64 columns at
        // a time (the score buffer is released after the second load). The
        // mask is a compile-time branch: the off-diagonal tiles (all but one
        // per row tile) carry no per-score compare or select.
        const bool diag = (j * kTile + kTile - 1 > row0);
        auto cols = [&](const uint32_t (&v)[32], int base, uint64_t& sum2, auto masked) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            // 2^(s*sigma*log2e - lse2) = 2^(fma(s, c, -lse2))
            float y0, y1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sc2,
                             lse2[(base + e) >> 1]),
                      y0, y1);
            float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
            if constexpr (decltype(masked)::value) {
              p0 = (kj <= row0 + base + e) ? p0 : 0.f;
              p1 = (kj <= row0 + base + e + 1) ? p1 : 0.f;
            }
            sum2 = f2_add(sum2, f2_pack(p0, p1));
          }
        };
        auto key_tile = [&](auto masked) {
          uint64_t acc[2] = {0ull, 0ull};
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t va[32], vb[32];
            tmem_ld32(ts + hh * 64, va);
            tmem_ld32(ts + hh * 64 + 32, vb);
            tmem_wait_ld();
            if (hh == 1) {
              tc_fence_before();
              mbar_arrive(s_free + sb);
            }
            cols(va, hh * 64, acc[0], masked);
            cols(vb, hh * 64 + 32, acc[1], masked);
          }
          float s0, s1;
          f2_unpack(f2_add(acc[0], acc[1]), s0, s1);
          return s0 + s1;
        };
        const float wsum = diag ? key_tile(BoolC<true>{}) : key_tile(BoolC<false>{});
        if (kj < L) wrow[kj] = wsum;
      }
      mbar_arrive(q_free + buf);   // done with this tile's LSEs
      kc += nkv;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
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

// Streaming multiprocessors of the current device (queried once per device).
int sm_count() {
  thread_local int cached_dev = -1, cached = 0;   // per host thread: no shared state
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev != cached_dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached = n;
    cached_dev = dev;
  }
  return cached;
}

template <bool REUSE, bool LSE>
cudaError_t launch_fa(const PrefillArgs& a, cudaStream_t st) {
  using SM = Fa2Smem<REUSE>;
  alignas(64) CUtensorMap tq, tk, tv;
  if (!make_maps(a, &tq, &tk, &tv, SM::KC)) return cudaErrorInvalidValue;
  alignas(64) CUtensorMap to;
  if (!encode_tmap_2d_bf16(&to, a.out, 128, static_cast<uint64_t>(a.B) * a.Hq * a.N, 64, kTile,
                           true))
    return cudaErrorInvalidValue;
  auto kern = k_prefill_fa2<REUSE, LSE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SM::SMEM));
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (shared memory and TMEM allow one), each
  // taking every gridDim-th tile
  const int tiles = a.B * a.Hq * a.nT;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidValue;
  const int grid = tiles < sms ? tiles : sms;
  kern<<<grid, fa_threads<REUSE>(), SM::SMEM, st>>>(tq, tk, tv, to, a);
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
  if (!make_maps(a, &tq, &tk, nullptr, kTile)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k_prefill_weights,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kWtSmemBytes));
  if (e != cudaSuccess) return e;
  const int tiles = a.B * a.Hq * a.nT;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidValue;
  k_prefill_weights<<<tiles < sms ? tiles : sms, kWtThreads, kWtSmemBytes, st>>>(tq, tk, a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_reuse(const PrefillArgs& a, int head_dim, cudaStream_t st) {
  if (head_dim != 128) return cudaErrorNotSupported;
  if (a.pooled && a.G >= 2 && a.G % 2 == 0) {
    // pooled sets: two query heads of a KV head per CTA, sharing every gather
    alignas(64) CUtensorMap tq;
    if (!make_maps(a, &tq, nullptr, nullptr, PairSmem::KC)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_prefill_pair,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(PairSmem::SMEM));
    if (e != cudaSuccess) return e;
    k_prefill_pair<<<a.B * a.Hkv * (a.G / 2) * a.nT, kPairThreads, PairSmem::SMEM, st>>>(tq, a);
    return cudaGetLastError();
  }
  return launch_fa<true, false>(a, st);
}

}  // namespace kascade
