// topk.cu — exact Top-k of fp32 rows (Kascade anchor layers take an exact,
// head-aware Top-k; euno.news summary, Key Contributions and Methodology 2,
// 5). Rule: larger score first, lower index wins a tie, -0 == +0; output
// ascending positions.
//
// One CTA per row (512 threads, two per SM; 256 threads, four per SM, for
// the many short rows of the prefill tiles); scores become order-preserving
// uint32 keys on the fly.
//   1. bracket: an evenly spaced sample of the row (len/16 keys, 2048..8192)
//      is staged in shared memory; two histogram passes over it give the
//      22-bit key prefixes at sample ranks rc -/+ margin (rc the expected
//      rank of the k-th key, margin four binomial standard deviations), i.e.
//      thresholds t_hi >= (k-th key) >= t_lo with high probability;
//   2. one coalesced pass over the row: a warp ballot per 32 positions gives
//      the bitmap of keys above t_hi (no atomics), and keys in [t_lo, t_hi]
//      are compacted into a shared candidate list;
//   3. if the bracket holds the k-th key, exact rank selection among the
//      candidates gives T; candidates > T join the "above" bitmap, == T the
//      "equal" bitmap. Otherwise (heavy ties, an unlucky sample) the exact
//      fallback runs 11/11/10-bit radix digit passes over the row;
//   4. ordered emission: a block scan over per-thread word runs gives each
//      thread its output offset; keys == T are taken in position order until
//      k positions are written.
// Prefill rows are the packed tile weights of one (sequence, head, tile):
// length L_t = min(N, 128(t+1)), k_t = min(k, L_t), -1 padding after k_t.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace kascade {
namespace {

// Candidate (key, position) pairs in shared memory: kCandCap for rows up to
// kShortRow keys (two CTAs per SM); longer rows take a larger pool (one CTA per
// SM) so that the per-warp lists do not overflow into the exact fallback.
constexpr int kCandCap = 4096;
constexpr int kShortRow = 32768;
constexpr int kMaxCandCap = 16384;
constexpr int kUnroll = 8;       // 32-position chunks in flight per warp
constexpr int kSampleCap = 8192; // evenly spaced sample used to bracket the k-th key
constexpr int kManyRows = 1024;  // rows from which short rows take 256-thread CTAs

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

// Inclusive block scan of one int per thread (NT threads).
template <int NT>
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
    int t = lane < NT / 32 ? warp_tot[lane] : 0;
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

// Visit the row in warp-owned blocks of 32*kUnroll consecutive positions;
// f(pos, valid, key) runs on every lane (warp-uniform control flow).
template <int NT, typename F>
__device__ __forceinline__ void for_row(const RowDesc& rd, bool& bad, F f) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int base = warp * 32 * kUnroll; base < rd.len; base += (NT / 32) * 32 * kUnroll) {
    float x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = base + 32 * u + lane;
      x[u] = j < rd.len ? __ldg(rd.ptr + j) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = base + 32 * u + lane;
      const bool valid = j < rd.len;
      bad |= valid && isnan(x[u]);
      f(j, valid, float_key(x[u]));
    }
  }
}

// Bin holding rank `need` (1 = largest) of an nb-bin histogram, counting from
// the top bin down; returns the bin and the count in the bins above it. Each
// of the NT threads owns nb / NT consecutive bins (highest first).
template <int NT>
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nb, int need, int* warp_tot,
                                         int* s_bin, int* s_above, int& bin, int& above) {
  const int per = nb / NT;
  const int top = nb - 1 - per * static_cast<int>(threadIdx.x);
  int local = 0;
  for (int q = 0; q < per; ++q) local += static_cast<int>(hist[top - q]);
  int run = block_incl_scan<NT>(local, warp_tot) - local;   // count above this thread's bins
  if (run < need && need <= run + local) {
    for (int q = 0; q < per; ++q) {
      const int h = static_cast<int>(hist[top - q]);
      if (need <= run + h) {
        *s_bin = top - q;
        *s_above = run;
        break;
      }
      run += h;
    }
  }
  __syncthreads();
  bin = *s_bin;
  above = *s_above;
  __syncthreads();
}

// Candidate i of the per-warp lists (list w holds count[w] keys at
// cand + w * warp_cap) in list order; pre[w] = keys in lists before w.
template <int NT>
__device__ __forceinline__ int cand_slot(const int* pre, int warp_cap, int i) {
  int w = 0;
#pragma unroll
  for (int q = 1; q < NT / 32; ++q) w += (i >= pre[q]) ? 1 : 0;
  return w * warp_cap + (i - pre[w]);
}

// select_rank over the per-warp candidate lists: all candidates lie in
// [t_lo, t_lo + span], so the digits are those of key - t_lo, from the top
// bit of span down in passes of at most 11 bits (one or two passes for a
// narrow bracket), each histogram built by one flat loop over the candidates.
template <int NT>
__device__ void select_rank_warp_lists(const uint32_t* cand, const int* pre, int total,
                                       int warp_cap, uint32_t t_lo, uint32_t span, int rank,
                                       uint32_t* hist, int* warp_tot, int* s_bin, int* s_above,
                                       uint32_t& key_out, int& greater) {
  const int nbits = span == 0u ? 1 : 32 - __clz(span);
  uint32_t prefix = 0, pmask = 0;
  int gt = 0;
  for (int top = nbits; top > 0;) {
    const int width = top > 11 ? 11 : top;
    const int sh = top - width;
    const int nb = 1 << width;
    for (int i = threadIdx.x; i < 2048; i += NT) hist[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < total; i += NT) {
      const uint32_t rel = cand[cand_slot<NT>(pre, warp_cap, i)] - t_lo;
      if ((rel & pmask) == prefix) atomicAdd(&hist[(rel >> sh) & (nb - 1)], 1u);
    }
    __syncthreads();
    int bin, above;
    find_bin<NT>(hist, nb < NT ? NT : nb, rank - gt, warp_tot, s_bin, s_above, bin, above);
    gt += above;
    prefix |= static_cast<uint32_t>(bin) << sh;
    pmask |= static_cast<uint32_t>(nb - 1) << sh;
    top = sh;
  }
  key_out = t_lo + prefix;
  greater = gt;
}

// Two sample quantiles at once, to 22-bit key resolution: the 22-bit key
// prefixes of the r_hi-th and r_lo-th largest sample keys (r_hi <= r_lo),
// from one 11-bit histogram of the sample and one of each boundary bin.
template <int NT>
__device__ void sample_bracket(const uint32_t* samp, int n, int r_hi, int r_lo, uint32_t* hist,
                               int* warp_tot, int* s_bin, int* s_above, uint32_t& p_hi,
                               uint32_t& p_lo) {
  uint32_t* h2 = hist + 2048;   // second histogram (second digit of the r_lo bin)
  for (int i = threadIdx.x; i < 4096; i += NT) hist[i] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += NT) atomicAdd(&hist[samp[i] >> 21], 1u);
  __syncthreads();
  int b_hi, a_hi, b_lo, a_lo;
  find_bin<NT>(hist, 2048, r_hi, warp_tot, s_bin, s_above, b_hi, a_hi);
  find_bin<NT>(hist, 2048, r_lo, warp_tot, s_bin, s_above, b_lo, a_lo);
  for (int i = threadIdx.x; i < 2048; i += NT) hist[i] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += NT) {
    const uint32_t key = samp[i];
    const uint32_t top = key >> 21, mid = (key >> 10) & 2047u;
    if (top == static_cast<uint32_t>(b_hi)) atomicAdd(&hist[mid], 1u);
    if (top == static_cast<uint32_t>(b_lo)) atomicAdd(&h2[mid], 1u);
  }
  __syncthreads();
  int m_hi, x_hi, m_lo, x_lo;
  find_bin<NT>(hist, 2048, r_hi - a_hi, warp_tot, s_bin, s_above, m_hi, x_hi);
  find_bin<NT>(h2, 2048, r_lo - a_lo, warp_tot, s_bin, s_above, m_lo, x_lo);
  p_hi = (static_cast<uint32_t>(b_hi) << 11) | static_cast<uint32_t>(m_hi);
  p_lo = (static_cast<uint32_t>(b_lo) << 11) | static_cast<uint32_t>(m_lo);
}

// NT threads per row. UNROLL: 32-position chunks per warp per step of the
// main pass (the next step's loads are in flight meanwhile); long rows run one
// CTA per SM with a deeper main pass, decode rows two CTAs per SM, the short
// prefill tile rows four.
template <int NT, int UNROLL, int MIN_BLOCKS>
__global__ void __launch_bounds__(NT, MIN_BLOCKS) k_topk(const __grid_constant__ TopkArgs a,
                                                         int words_cap, int cand_cap) {
  constexpr int kThreads = NT, kWarps = NT / 32;
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t sm[];
  uint32_t* hist = sm;                                                     // [2][2048]
  const int warp_cap = cand_cap / kWarps;                                  // per-warp list
  uint32_t* cand_key = hist + 4096;                                        // [cand_cap]
  int32_t* cand_pos = reinterpret_cast<int32_t*>(cand_key + cand_cap);     // [cand_cap]
  // the sample is only used before the candidates exist: it shares their space
  uint32_t* samp = cand_key;                                               // [kSampleCap]
  uint32_t* above = hist + 4096 + max(2 * cand_cap, kSampleCap);          // [words_cap]
  uint32_t* eqbm = above + words_cap;                                      // [words_cap]
  __shared__ int warp_tot[32];
  __shared__ int s_ncand, s_nabove, s_bin, s_above;
  __shared__ int s_wcount[kWarps];

  const int r = blockIdx.x;
  const RowDesc rd = row_desc(a, r);
  const int tid = threadIdx.x, lane = tid & 31;
  int32_t* out = a.idx_out + static_cast<size_t>(r) * a.k_stride;

  if (rd.k >= rd.len) {   // the whole prefix is selected
    for (int j = tid; j < a.k_stride; j += kThreads) out[j] = (j < rd.len) ? j : -1;
    if (a.sel_bits != nullptr) {
      const int Ws = (rd.len + 31) >> 5;
      for (int w = tid; w < Ws; w += kThreads) {
        const int rest = rd.len - 32 * w;
        a.sel_bits[static_cast<size_t>(r) * Ws + w] = rest >= 32 ? 0xFFFFFFFFu : (1u << rest) - 1u;
      }
    }
    return;
  }
  const int W = (rd.len + 31) >> 5;
  for (int w = tid; w < W; w += kThreads) above[w] = eqbm[w] = 0u;
  if (tid == 0) {
    s_ncand = 0;
    s_nabove = 0;
  }
  const int warp = tid >> 5;
  int c_gt = 0;
  bool bad = false;
  bool fused_ok = false;
  if (a.flist != nullptr) {
    // ---- fused anchor decode: select from the list the attention kernel
    // wrote (every key >= t_lo of the row) instead of reading the row. Keys
    // above t_hi are selected outright; the k-th key is found among those in
    // [t_lo, t_hi] (candidates, shared memory). Any miss (list overflow, the
    // k-th key outside the bracket, too many candidates) takes the full path
    // below over the row itself.
    __shared__ int s_fa, s_fc;
    if (tid == 0) {
      s_fa = 0;
      s_fc = 0;
    }
    __syncthreads();
    const uint2 br = a.bracket[r];
    {
      // the row's sub-lists, one per (split, warp) of the attention kernel,
      // taken by the warps in turn
      const int nsub = a.fsplits * a.fwarps;
      const int cap_sub = a.fchunk / a.fwarps;
      const uint2* rl = a.flist + static_cast<size_t>(r) * a.fsplits * a.fchunk;
      const unsigned int* rc = a.fcount + static_cast<size_t>(r) * nsub;
      int my_above = 0;
      // each warp's sub-list lengths in one round of loads (lane i holds the
      // length of the warp's i-th sub-list), then every sub-list in batches
      // of 4 entries per lane whose loads are all issued before any use
      constexpr int kBatch = 4;
      for (int sub0 = warp; sub0 < nsub; sub0 += 32 * kWarps) {
        const int my_sub = sub0 + lane * kWarps;
        const int my_cnt = my_sub < nsub ? min(static_cast<int>(rc[my_sub]), cap_sub) : 0;
        for (int i = 0; i < 32 && sub0 + i * kWarps < nsub; ++i) {
          const int sub = sub0 + i * kWarps;
          const int cnt = __shfl_sync(0xffffffffu, my_cnt, i);
          const uint2* list = rl + static_cast<size_t>(sub) * cap_sub;
          for (int e0 = 0; e0 < cnt; e0 += 32 * kBatch) {
            uint2 kp[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
              kp[u] = list[min(e0 + u * 32 + lane, cnt - 1)];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
              const bool valid = e0 + u * 32 + lane < cnt;
              const int p = static_cast<int>(kp[u].y);
              const bool is_above = valid && kp[u].x > br.y;
              const bool is_mid = valid && !is_above;
              if (is_above) {
                atomicOr(&above[p >> 5], 1u << (p & 31));
                ++my_above;
              }
              // candidates: one slot reservation per warp
              const unsigned int mm = __ballot_sync(0xffffffffu, is_mid);
              if (mm != 0u) {
                int base = 0;
                if (lane == __ffs(mm) - 1) base = atomicAdd(&s_fc, __popc(mm));
                base = __shfl_sync(0xffffffffu, base, __ffs(mm) - 1);
                if (is_mid) {
                  const int slot = base + __popc(mm & ((1u << lane) - 1u));
                  if (slot < cand_cap) {
                    cand_key[slot] = kp[u].x;
                    cand_pos[slot] = p;
                  }
                }
              }
            }
          }
        }
      }
      if (my_above) atomicAdd(&s_fa, my_above);
      __syncthreads();
      const int n_above = s_fa, n_mid = s_fc;
      if (n_mid <= cand_cap && n_above < rd.k && n_above + n_mid >= rd.k) {
        __shared__ int s_fpre[kWarps + 1];
        for (int w = tid; w <= kWarps; w += kThreads) s_fpre[w] = w == 0 ? 0 : n_mid;
        __syncthreads();
        uint32_t T;
        int cg;
        // one flat list (list 0 holds every candidate)
        select_rank_warp_lists<NT>(cand_key, s_fpre, n_mid, cand_cap, br.x, br.y - br.x,
                                   rd.k - n_above, hist, warp_tot, &s_bin, &s_above, T, cg);
        c_gt = n_above + cg;
        for (int i = tid; i < n_mid; i += kThreads) {
          const uint32_t key = cand_key[i];
          const int p = cand_pos[i];
          if (key > T) atomicOr(&above[p >> 5], 1u << (p & 31));
          else if (key == T) atomicOr(&eqbm[p >> 5], 1u << (p & 31));
        }
        fused_ok = true;
      }
    }
    __syncthreads();
    if (!fused_ok) {
      for (int w = tid; w < W; w += kThreads) above[w] = 0u;
      if (tid == 0) {
        s_ncand = 0;
        s_nabove = 0;
      }
    }
    __syncthreads();
  }
  if (!fused_ok) {

  // ---- 1. bracket the k-th key from an evenly spaced sample -------------
  const int S = min(rd.len, max(2048, min(kSampleCap, rd.len / 16)));
  // The sample is S / 32 evenly spaced runs of 32 consecutive keys, one
  // 128-byte line per run, so that sampling costs whole lines rather than one
  // DRAM sector per sample (the exact selection below does not depend on how
  // the sample was drawn; a poor sample only costs the fallback).
  {
    const int runs = S / 32;
    const float step = static_cast<float>(rd.len - 32) / static_cast<float>(max(runs - 1, 1));
    for (int u0 = 0; u0 < S; u0 += 16 * kThreads) {   // 16 loads in flight per thread
      float v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int u = u0 + q * kThreads + tid;
        const int j = min(rd.len - 1, __float2int_rd(static_cast<float>(u >> 5) * step) + (u & 31));
        v[q] = u < S ? __ldg(rd.ptr + j) : 0.f;
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int u = u0 + q * kThreads + tid;
        if (u < S) samp[u] = float_key(v[q]);
      }
    }
  }
  __syncthreads();
  const float rc = static_cast<float>(rd.k) * S / rd.len;   // expected sample rank
  const float margin = 4.f * sqrtf(rc) + 16.f;
  const int r_hi = static_cast<int>(floorf(rc - margin));
  const int r_lo = static_cast<int>(ceilf(rc + margin));
  // above: 22-bit prefix > p_hi; candidates: p_lo <= prefix <= p_hi
  uint32_t t_hi = 0xFFFFFFFFu, t_lo = 0u;
  {
    uint32_t p_hi, p_lo;
    sample_bracket<NT>(samp, S, max(r_hi, 1), min(r_lo, S), hist, warp_tot, &s_bin, &s_above,
                       p_hi, p_lo);
    if (r_hi >= 1) t_hi = (p_hi << 10) | 1023u;
    if (r_lo <= S) t_lo = p_lo << 10;
  }

  // ---- 2. one pass: "above" bitmap by ballot, candidates in [t_lo, t_hi] --
  // Each warp owns blocks of 32*UNROLL consecutive positions and appends its
  // candidates to its own shared list (count kept in a register).
  uint32_t* wkey = cand_key + warp * warp_cap;
  int32_t* wpos = cand_pos + warp * warp_cap;
  const uint32_t span = t_hi - t_lo;
  int wcount = 0, my_above = 0;
  // the next block's scores are loaded before this block is processed
  float xn[UNROLL];
  {
    const int base = warp * 32 * UNROLL;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int j = base + 32 * u + lane;
      xn[u] = j < rd.len ? __ldg(rd.ptr + j) : 0.f;
    }
  }
  for (int base = warp * 32 * UNROLL; base < rd.len; base += kWarps * 32 * UNROLL) {
    float x[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) x[u] = xn[u];
    const int nbase = base + kWarps * 32 * UNROLL;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int j = nbase + 32 * u + lane;
      xn[u] = j < rd.len ? __ldg(rd.ptr + j) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int j = base + 32 * u + lane;
      const bool valid = j < rd.len;
      bad |= x[u] != x[u];
      const uint32_t key = float_key_fast(x[u]);
      const unsigned int ba = __ballot_sync(0xffffffffu, valid && key > t_hi);
      const bool in = valid && (key - t_lo) <= span;
      const unsigned int bi = __ballot_sync(0xffffffffu, in);
      if (lane == 0 && (base + 32 * u) < rd.len) above[(base >> 5) + u] = ba;
      my_above += __popc(ba);
      if (in) {
        const int p = wcount + __popc(bi & ((1u << lane) - 1u));
        if (p < warp_cap) {
          wkey[p] = key;
          wpos[p] = j;
        }
      }
      wcount += __popc(bi);
    }
  }
  if (lane == 0) {
    s_wcount[warp] = wcount;
    atomicAdd(&s_nabove, my_above);
    if (wcount > warp_cap) atomicAdd(&s_ncand, 1);   // overflow marker
  }
  if (__syncthreads_or(bad) && tid == 0) report_error(a.err, KASCADE_ERR_BAD_INPUT, 0x401);
  int n_cand = 0;
  for (int w = 0; w < kWarps; ++w) n_cand += s_wcount[w];
  const int n_above = s_nabove;
  const bool overflow = s_ncand != 0;
  if (!overflow && n_above < rd.k && n_above + n_cand >= rd.k) {
    // ---- 3. exact k-th key among the candidates -------------------------
    uint32_t T;
    int cg;
    __shared__ int s_pre[kWarps + 1];
    if (tid == 0) {
      int acc = 0;
      for (int w = 0; w < kWarps; ++w) {
        s_pre[w] = acc;
        acc += s_wcount[w];
      }
      s_pre[kWarps] = acc;
    }
    __syncthreads();
    select_rank_warp_lists<NT>(cand_key, s_pre, n_cand, warp_cap, t_lo, span, rd.k - n_above,
                               hist, warp_tot, &s_bin, &s_above, T, cg);
    c_gt = n_above + cg;
    for (int i = tid; i < n_cand; i += kThreads) {
      const int slot = cand_slot<NT>(s_pre, warp_cap, i);
      const uint32_t key = cand_key[slot];
      const int p = cand_pos[slot];
      if (key > T) atomicOr(&above[p >> 5], 1u << (p & 31));
      else if (key == T) atomicOr(&eqbm[p >> 5], 1u << (p & 31));
    }
    __syncthreads();
  } else {
    // ---- fallback (heavy ties or an unlucky sample): exact digit passes ---
    for (int w = tid; w < W; w += kThreads) above[w] = eqbm[w] = 0u;
    uint32_t prefix = 0, pmask = 0;
    c_gt = 0;
    for (int d = 0; d < 3; ++d) {
      const int nb = d < 2 ? 2048 : 1024;
      const int sh = d == 0 ? 21 : (d == 1 ? 10 : 0);
      for (int i = tid; i < nb; i += kThreads) hist[i] = 0u;
      __syncthreads();
      for_row<NT>(rd, bad, [&](int, bool valid, uint32_t key) {
        hist_add(hist, valid && (key & pmask) == prefix, (key >> sh) & (nb - 1));
      });
      __syncthreads();
      int bin, ab;
      find_bin<NT>(hist, nb, rd.k - c_gt, warp_tot, &s_bin, &s_above, bin, ab);
      c_gt += ab;
      prefix |= static_cast<uint32_t>(bin) << sh;
      pmask |= static_cast<uint32_t>(nb - 1) << sh;
    }
    const uint32_t T = prefix;
    for_row<NT>(rd, bad, [&](int j, bool valid, uint32_t key) {
      const unsigned int ba = __ballot_sync(0xffffffffu, valid && key > T);
      const unsigned int be = __ballot_sync(0xffffffffu, valid && key == T);
      if (lane == 0 && j < rd.len) {
        above[j >> 5] = ba;
        eqbm[j >> 5] = be;
      }
    });
    __syncthreads();
  }
  }   // full path

  // ---- 4. ordered emission ----------------------------------------------
  const int need_eq = rd.k - c_gt;
  const int per = (W + kThreads - 1) / kThreads;
  const int w0 = min(W, tid * per), w1 = min(W, w0 + per);
  int ca = 0, ce = 0;
  for (int w = w0; w < w1; ++w) {
    ca += __popc(above[w]);
    ce += __popc(eqbm[w]);
  }
  int pa = block_incl_scan<NT>(ca, warp_tot) - ca;
  int pe = block_incl_scan<NT>(ce, warp_tot) - ce;
  for (int w = w0; w < w1; ++w) {
    const uint32_t ab = above[w], eb = eqbm[w];
    uint32_t u = ab | eb;
    uint32_t sel = 0u;   // the positions of this word that were emitted
    while (u) {
      const int bit = __ffs(u) - 1;
      u &= u - 1;
      const int pos = w * 32 + bit;
      if ((ab >> bit) & 1u) {
        const int o = pa + min(pe, need_eq);
        if (o < rd.k) {
          out[o] = pos;
          sel |= 1u << bit;
        }
        ++pa;
      } else {
        if (pe < need_eq && pa + pe < rd.k) {
          out[pa + pe] = pos;
          sel |= 1u << bit;
        }
        ++pe;
      }
    }
    if (a.sel_bits != nullptr) a.sel_bits[static_cast<size_t>(r) * W + w] = sel;
  }
  for (int j = rd.k + tid; j < a.k_stride; j += kThreads) out[j] = -1;
}

// ------------------------------------------------------------------------
// Fused anchor decode, step 1: the sample bracket of every logit row, taken
// before the attention kernel so that it can file each row's candidates as
// it computes the logits. The sample is k_topk's: `runs` evenly spaced runs
// of 32 consecutive keys per row (every key of a row shorter than 2048).
//   k_anchor_sample : the sample logits sigma q.k of one (sequence, KV head)
//                     for all G heads of the group at once (each K row read
//                     once), a few runs per CTA, as order-preserving keys;
//   k_anchor_bracket: per row, the two sample quantiles -> (t_lo, t_hi).
// The logits here are fp32 CUDA-core dot products: only the bracket depends
// on them; the selection is made on the attention kernel's own values.
// ------------------------------------------------------------------------
struct SampleGeom {
  int S;        // sample size (a multiple of 32, or the whole row)
  int runs;     // runs of 32 keys
  bool whole;   // the whole row is the sample
  float step;   // run spacing
};

__host__ __device__ inline SampleGeom sample_geom(int len) {
  SampleGeom g;
  g.whole = len < 2048;
  const int s = len / 16 > 2048 ? len / 16 : 2048;
  g.S = g.whole ? len : ((s < kSampleCap ? s : kSampleCap) / 32) * 32;
  g.runs = (g.S + 31) / 32;
  g.step = g.whole ? 32.f : static_cast<float>(len - 32) / static_cast<float>(g.runs > 1 ? g.runs - 1 : 1);
  return g;
}

struct SampleArgs {
  const __nv_bfloat16* q;   // [B,Hq,D]
  const __nv_bfloat16* k;   // [B,Hkv,N,D]
  uint32_t* samp;           // [B*Hq][S] sample keys
  int Hq, Hkv, N, S_stride;
  float scale;
  int16_t heads[kMaxQHeads];   // heads[g*G + slot]
};

constexpr int kSampWarps = 4, kSampRunsPerWarp = 2;

// One CTA: kSampWarps * kSampRunsPerWarp runs of one (sequence, KV head).
// A warp reads a run as one contiguous block: lane l holds 16-byte chunk
// l % CH of key row l / CH of each group of RPI rows (coalesced loads, all
// issued before the arithmetic); the CH lanes of a row reduce their partial
// dot products (G heads at once) by shuffles.
template <int D, int G>
__global__ void __launch_bounds__(kSampWarps * 32) k_anchor_sample(const __grid_constant__ SampleArgs a) {
  pdl_wait();
  pdl_trigger();
  constexpr int CH = D / 8, RPI = 32 / CH, NI = 32 / RPI;
  const int unit = blockIdx.y;
  const int b = unit / a.Hkv, g = unit % a.Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cc = lane % CH, sub = lane / CH;
  const int len = a.N;
  const SampleGeom sg = sample_geom(len);
  float qv[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(
                              a.q + (static_cast<size_t>(b) * a.Hq + a.heads[g * G + h]) * D) + cc);
    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(p2[e]);
      qv[h][2 * e] = f.x;
      qv[h][2 * e + 1] = f.y;
    }
  }
  const uint4* kb = reinterpret_cast<const uint4*>(a.k + static_cast<size_t>(unit) * a.N * D);
  const int run0 = (blockIdx.x * kSampWarps + warp) * kSampRunsPerWarp;
  for (int rr = 0; rr < kSampRunsPerWarp; ++rr) {
    const int run = run0 + rr;
    if (run >= sg.runs) break;
    const int start = sg.whole ? 32 * run : min(len - 32, __float2int_rd(static_cast<float>(run) * sg.step));
    uint4 w[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i)
      w[i] = __ldg(kb + static_cast<size_t>(min(start + i * RPI + sub, len - 1)) * CH + cc);
    // partial dot products over this lane's 8 dimensions, two at a time
    float part[G][NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&w[i]);
      uint64_t f[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(p2[e]);
        f[e] = f2_pack(x.x, x.y);
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        uint64_t acc = f2_pack(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc = f2_fma(f[e], f2_pack(qv[h][2 * e], qv[h][2 * e + 1]), acc);
        float lo, hi;
        f2_unpack(acc, lo, hi);
        part[h][i] = lo + hi;
      }
    }
    // reduce-scatter over the CH lanes of each row: at every step a lane
    // keeps half of its values and adds the partner's copy of that half, so
    // after log2(CH) steps lane cc holds the full sum of load i = ri(cc)
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int half = NI / 2; half >= 1; half >>= 1) {
        const bool upper = (cc & half) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
          const float send = upper ? part[h][j] : part[h][j + half];
          const float keep = upper ? part[h][j + half] : part[h][j];
          part[h][j] = keep + __shfl_xor_sync(0xffffffffu, send, half);
        }
      }
    }
    // lane cc now owns load index i = cc (the bit of `half` chose the upper
    // half at each step); its row is start + cc * RPI + sub
    {
      const int i = cc;
      const int u = 32 * run + i * RPI + sub;   // sample slot
      if (u < sg.S && start + i * RPI + sub < len) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          a.samp[(static_cast<size_t>(b) * a.Hq + a.heads[g * G + h]) * a.S_stride + u] =
              float_key(part[h][0] * a.scale);
      }
    }
  }
}

constexpr int kBrThreads = 512;

// One CTA per row: the two quantiles of its sample keys (as in k_topk).
__global__ void __launch_bounds__(kBrThreads) k_anchor_bracket(const uint32_t* __restrict__ samp,
                                                               int S_stride, int N, int topk,
                                                               uint2* __restrict__ bracket) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t sm[];
  uint32_t* hist = sm;            // [2][2048]
  uint32_t* ss = sm + 4096;       // [kSampleCap]
  __shared__ int warp_tot[32];
  __shared__ int s_bin, s_above;
  const int r = blockIdx.x, tid = threadIdx.x;
  const int len = N, k = min(topk, N);
  if (k >= len) {   // every key is selected (k_topk returns early)
    if (tid == 0) bracket[r] = make_uint2(0u, 0xFFFFFFFFu);
    return;
  }
  const SampleGeom sg = sample_geom(len);
  const int S = sg.S;
  const uint32_t* row = samp + static_cast<size_t>(r) * S_stride;
  for (int u = tid; u < S; u += kBrThreads) ss[u] = __ldg(row + u);
  __syncthreads();
  const float rc = static_cast<float>(k) * S / len;   // expected sample rank
  const float margin = 4.f * sqrtf(rc) + 16.f;
  const int r_hi = static_cast<int>(floorf(rc - margin));
  const int r_lo = static_cast<int>(ceilf(rc + margin));
  uint32_t p_hi, p_lo;
  sample_bracket<kBrThreads>(ss, S, max(r_hi, 1), min(r_lo, S), hist, warp_tot, &s_bin,
                             &s_above, p_hi, p_lo);
  if (tid == 0) {
    const uint32_t t_hi = r_hi >= 1 ? ((p_hi << 10) | 1023u) : 0xFFFFFFFFu;
    const uint32_t t_lo = r_lo <= S ? (p_lo << 10) : 0u;
    bracket[r] = make_uint2(t_lo, t_hi);
  }
}

template <int D, int G>
cudaError_t launch_sample_t(const SampleArgs& a, int units, int runs, cudaStream_t st) {
  const int per_cta = kSampWarps * kSampRunsPerWarp;
  return launch_pdl(k_anchor_sample<D, G>, dim3((runs + per_cta - 1) / per_cta, units),
                    dim3(kSampWarps * 32), 0, st, a);
}

}  // namespace

int anchor_sample_stride(int N) { return sample_geom(N).S; }

cudaError_t launch_anchor_bracket(const void* q, const void* k, const int16_t* heads, int B,
                                  int Hq, int Hkv, int N, int d, int topk, float scale,
                                  uint32_t* samp, uint2* bracket, cudaStream_t st) {
  const int rows = B * Hq;
  if (rows <= 0) return cudaSuccess;
  const int G = Hq / Hkv;
  const SampleGeom sg = sample_geom(N);
  if (topk < N) {
    SampleArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k = static_cast<const __nv_bfloat16*>(k);
    a.samp = samp;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.N = N;
    a.S_stride = sg.S;
    a.scale = scale;
    for (int h = 0; h < Hq; ++h) a.heads[h] = heads[h];
    const int units = B * Hkv;
    cudaError_t e = cudaErrorInvalidValue;
    if (d == 128) {
      if (G == 1) e = launch_sample_t<128, 1>(a, units, sg.runs, st);
      if (G == 2) e = launch_sample_t<128, 2>(a, units, sg.runs, st);
      if (G == 4) e = launch_sample_t<128, 4>(a, units, sg.runs, st);
      if (G == 8) e = launch_sample_t<128, 8>(a, units, sg.runs, st);
    } else if (d == 64) {
      if (G == 1) e = launch_sample_t<64, 1>(a, units, sg.runs, st);
      if (G == 2) e = launch_sample_t<64, 2>(a, units, sg.runs, st);
      if (G == 4) e = launch_sample_t<64, 4>(a, units, sg.runs, st);
      if (G == 8) e = launch_sample_t<64, 8>(a, units, sg.runs, st);
    }
    if (e != cudaSuccess) return e;
  }
  const size_t smem = (4096 + kSampleCap) * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(k_anchor_bracket, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(k_anchor_bracket, dim3(rows), dim3(kBrThreads), smem, st,
                    static_cast<const uint32_t*>(samp), sg.S, N, topk, bracket);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  const int words_cap = (a.n + 31) / 32;
  // shared memory: histogram, candidate pool (also holding the sample first),
  // two row bitmaps. Long rows first try a pool that keeps two CTAs per SM,
  // else take one CTA per SM with a larger pool.
  const size_t fixed = 4096 * sizeof(uint32_t) + 2 * static_cast<size_t>(words_cap) * sizeof(uint32_t);
  auto smem_for = [&](int cap) {
    const int region = 2 * cap > kSampleCap ? 2 * cap : kSampleCap;
    return fixed + static_cast<size_t>(region) * sizeof(uint32_t);
  };
  constexpr size_t kTwoPerSm = 110 * 1024, kOnePerSm = 220 * 1024;
  int cand_cap = kCandCap;
  bool one_per_sm = false;
  if (a.n > kShortRow) {
    auto fit = [&](size_t budget) {
      int cap = 0;
      if (budget > fixed) cap = static_cast<int>((budget - fixed) / (2 * sizeof(uint32_t)));
      cap = (cap < kMaxCandCap ? cap : kMaxCandCap) / 512 * 512;
      return cap;
    };
    cand_cap = fit(kTwoPerSm);
    if (cand_cap < 6144) {   // 384 per warp: room for the long-row bracket
      cand_cap = fit(kOnePerSm);
      one_per_sm = true;
    }
    if (cand_cap < kCandCap) cand_cap = kCandCap;
  }
  const size_t smem = smem_for(cand_cap);
  if (smem > kOnePerSm) return cudaErrorNotSupported;
  // Many short rows (the prefill tiles: 32 heads x 128 tiles at N = 16384)
  // run many waves of CTAs whose time goes to barriers and load latency, not
  // to bandwidth: 256-thread CTAs, four per SM (same registers per thread,
  // 52 KB of shared memory each at N = 16384), keep twice the rows in flight.
  const bool small = !one_per_sm && a.n <= kShortRow / 2 && a.rows >= kManyRows;
  auto kern = one_per_sm ? k_topk<512, 32, 1>
                         : (small ? k_topk<256, kUnroll, 4> : k_topk<512, kUnroll, 2>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(a.rows), dim3(small ? 256 : 512), smem, st, a, words_cap,
                    cand_cap);
}

}  // namespace kascade
