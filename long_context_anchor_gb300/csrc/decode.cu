// decode.cu — decode attention for one query per sequence (Kascade anchor
// and reuse layers; euno.news summary, Methodology 2-3).
//
//   k_decode_dense_bf16   split-K flash-decode over all N keys of one
//                         (sequence, KV head). A producer warp streams K/V
//                         tiles into shared memory with TMA (128-byte
//                         swizzle, mbarrier pipeline); consumer warps run the
//                         G query heads of the group together as mma.sync
//                         m16n8k16 tiles (keys x heads), online softmax in
//                         fp32, and (anchor layers) spill the scaled logits
//                         sigma*q.k for the Top-k selection.
//   k_build_union_plan    merges the G per-head index sets of one KV head
//                         into one ascending list of keys with a head mask.
//   k_decode_union_bf16   reuse layer: gathers only the planned K/V rows
//                         (16-byte cp.async into the same swizzled layout)
//                         and runs the same tile math with per-(key, head)
//                         masking, so a row shared by several heads of a
//                         group is read once.
//   k_decode_generic      CUDA-core path for fp32 inputs.
// The split kernels finish with a last-arriving-CTA merge of the split
// partials (log-sum-exp combine), so a layer is one launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"

namespace kascade {

namespace {

constexpr int kPlanCap = kPlanCapEntries;   // plan entries of one reuse CTA (shared staging)

#define kNegInf (-CUDART_INF_F)
constexpr float kLn2 = 0.6931471805599453f;   // log2-domain maxima back to logit units

// ------------------------------------------------------------------------
// Consumer math on one 16-key slice held in swizzled shared memory. Thread
// (gid = lane/4, c4 = lane%4) owns heads 2*c4, 2*c4+1 and keys gid, gid+8 of
// the slice's score tile, and output dims 16*mt+gid(+8) of those two heads.
// ------------------------------------------------------------------------
template <int D>
struct WarpState {
  float m[2];
  float l[2];
  float o[D / 16][4];
};

template <int D>
__device__ __forceinline__ void warp_state_init(WarpState<D>& st) {
  st.m[0] = st.m[1] = kNegInf;
  st.l[0] = st.l[1] = 0.f;
#pragma unroll
  for (int i = 0; i < D / 16; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.f;
}

// Scores of the 16 keys of a slice against the (up to 8) group heads:
// sc[0]=(key gid, head 2c4) sc[1]=(gid, 2c4+1) sc[2]=(gid+8, 2c4) sc[3]=(gid+8, 2c4+1).
template <int D>
__device__ __forceinline__ void slice_scores(uint32_t kbase, int rows, int row0,
                                             const uint32_t (&qf)[D / 16][2], float (&sc)[4]) {
  const int lane = threadIdx.x & 31;
  const int mi = lane >> 3, r = lane & 7;
  const int row = row0 + (mi & 1) * 8 + r;
  float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(kbase + sw128_offset(rows, row, 2 * kk + (mi >> 1)), a0, a1, a2, a3);
    if (kk & 1)
      mma_bf16_16816(acc1, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
    else
      mma_bf16_16816(acc0, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) sc[i] = acc0[i] + acc1[i];
}

// Online-softmax update with log2-domain scores x (masked entries -inf),
// then O^T += V^T P^T on the tensor cores.
template <int D>
__device__ __forceinline__ void slice_softmax_pv(WarpState<D>& st, const float (&x)[4],
                                                 uint32_t vbase, int rows, int row0) {
  const int lane = threadIdx.x & 31;
  float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
  }
  const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
  const float al0 = (mn0 == kNegInf) ? 1.f : fast_exp2(st.m[0] - mn0);
  const float al1 = (mn1 == kNegInf) ? 1.f : fast_exp2(st.m[1] - mn1);
  const float mu0 = (mn0 == kNegInf) ? 0.f : mn0;
  const float mu1 = (mn1 == kNegInf) ? 0.f : mn1;
  const float p0 = fast_exp2(x[0] - mu0), p1 = fast_exp2(x[1] - mu1);
  const float p2 = fast_exp2(x[2] - mu0), p3 = fast_exp2(x[3] - mu1);
  st.l[0] = st.l[0] * al0 + p0 + p2;
  st.l[1] = st.l[1] * al1 + p1 + p3;
  st.m[0] = mn0;
  st.m[1] = mn1;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    st.o[mt][0] *= al0;
    st.o[mt][1] *= al1;
    st.o[mt][2] *= al0;
    st.o[mt][3] *= al1;
  }
  // P (keys x heads) -> P^T fragments (heads x keys) for the B operand.
  const uint32_t b0 = movmatrix_t(pack_bf16(p0, p1));
  const uint32_t b1 = movmatrix_t(pack_bf16(p2, p3));
  const int mi = lane >> 3, r = lane & 7;
  const int row = row0 + (mi >> 1) * 8 + r;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4_t(vbase + sw128_offset(rows, row, 2 * mt + (mi & 1)), a0, a1, a2, a3);
    mma_bf16_16816(st.o[mt], a0, a1, a2, a3, b0, b1);
  }
}

// q fragments (B operand of keys x heads): qf[kk] = q[head gid][16kk + 2c4 (+8)].
template <int D>
__device__ __forceinline__ void load_q_frags(const DecodeArgs& a, int b, int g,
                                             uint32_t (&qf)[D / 16][2]) {
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2, c4 = lane & 3;
  const bool ok = gid < a.G;
  const int hq = ok ? a.heads[g * a.G + gid] : 0;
  const uint32_t* qrow =
      reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.q) +
                                        (static_cast<size_t>(b) * a.Hq + hq) * D);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    qf[kk][0] = ok ? __ldg(qrow + 8 * kk + c4) : 0u;
    qf[kk][1] = ok ? __ldg(qrow + 8 * kk + 4 + c4) : 0u;
  }
}

// Merge the consumer warps' states through shared memory, write this CTA's
// partial (or the final output when there is one split), and let the last
// CTA of the (sequence, KV head) merge all splits. `scratch` must hold
// (16 + 8*D) * n_consumers + 16 + 24 * S floats.
template <int D>
__device__ void finish_cta(const DecodeArgs& a, WarpState<D>& st, int cw, int n_consumers,
                           float* scratch, int b, int g, int split) {
  __shared__ unsigned int s_last;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2, c4 = lane & 3;
  // sum l across the 8 lanes that share a head pair
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], off);
    st.l[1] += __shfl_xor_sync(0xffffffffu, st.l[1], off);
  }
  // scratch layout: m[W][8], l[W][8], o[W][8][D], cm[8], cl[8]
  float* sm = scratch;
  float* sl = scratch + n_consumers * 8;
  float* so = scratch + n_consumers * 16;
  float* cm = so + n_consumers * 8 * D;
  float* cl = cm + 8;
  if (cw >= 0) {
    if (gid == 0) {
      sm[cw * 8 + 2 * c4] = st.m[0];
      sm[cw * 8 + 2 * c4 + 1] = st.m[1];
      sl[cw * 8 + 2 * c4] = st.l[0];
      sl[cw * 8 + 2 * c4 + 1] = st.l[1];
    }
    float* base = so + (cw * 8) * D;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      base[(2 * c4) * D + 16 * mt + gid] = st.o[mt][0];
      base[(2 * c4 + 1) * D + 16 * mt + gid] = st.o[mt][1];
      base[(2 * c4) * D + 16 * mt + gid + 8] = st.o[mt][2];
      base[(2 * c4 + 1) * D + 16 * mt + gid + 8] = st.o[mt][3];
    }
  }
  __syncthreads();
  const int G = a.G;
  const int unit = b * a.Hkv + g;
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float M = kNegInf;
    for (int w = 0; w < n_consumers; ++w) M = fmaxf(M, sm[w * 8 + h]);
    float L = 0.f;
    for (int w = 0; w < n_consumers; ++w) {
      const float mw = sm[w * 8 + h];
      if (mw != kNegInf) L += fast_exp2(mw - M) * sl[w * 8 + h];
    }
    cm[h] = M;
    cl[h] = L;
    if (a.S == 1 && a.row_stat != nullptr)   // the row's softmax statistics, in logit units
      a.row_stat[static_cast<size_t>(b) * a.Hq + a.heads[g * G + h]] =
          make_float2(M * kLn2, L > 0.f ? 1.f / L : 0.f);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int h = e / D, dd = e % D;
    const float M = cm[h];
    float acc = 0.f;
    for (int w = 0; w < n_consumers; ++w) {
      const float mw = sm[w * 8 + h];
      if (mw != kNegInf) acc += fast_exp2(mw - M) * so[(w * 8 + h) * D + dd];
    }
    const int hq = a.heads[g * G + h];
    if (a.S == 1) {
      const float L = cl[h];
      const float y = L > 0.f ? acc / L : 0.f;
      static_cast<__nv_bfloat16*>(a.out)[(static_cast<size_t>(b) * a.Hq + hq) * D + dd] =
          __float2bfloat16_rn(y);
    } else {
      float* pp = a.part + ((static_cast<size_t>(b) * a.Hq + hq) * a.S + split) * (D + 4);
      pp[4 + dd] = acc;
      if (dd == 0) {
        pp[0] = M;
        pp[1] = cl[h];
      }
    }
  }
  if (a.S == 1) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int prev = atomicAdd(&a.counters[unit], 1u);
    s_last = (prev == static_cast<unsigned int>(a.S - 1)) ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // Final merge over splits: weights w_s = 2^(m_s - M) / L per head. Every
  // split's (m, l) is loaded by its own thread first (one round of global
  // loads instead of a chain of them), then summed in split order.
  float* wts = cl + 8;           // [G][S]
  float* pm = wts + G * a.S;     // [G][S] split maxima
  float* pl = pm + G * a.S;      // [G][S] split sums
  for (int e = threadIdx.x; e < G * a.S; e += blockDim.x) {
    const int h = e / a.S, s = e % a.S;
    const float* pp = a.part + ((static_cast<size_t>(b) * a.Hq + a.heads[g * G + h]) * a.S + s) * (D + 4);
    pm[e] = __ldcg(pp);
    pl[e] = __ldcg(pp + 1);
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float M = kNegInf;
    for (int s = 0; s < a.S; ++s) M = fmaxf(M, pm[h * a.S + s]);
    float L = 0.f;
    for (int s = 0; s < a.S; ++s) {
      const float ms = pm[h * a.S + s];
      const float w = (ms == kNegInf) ? 0.f : fast_exp2(ms - M);
      wts[h * a.S + s] = w;
      L += w * pl[h * a.S + s];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int s = 0; s < a.S; ++s) wts[h * a.S + s] *= inv;
    if (a.row_stat != nullptr)   // the row's softmax statistics, in logit units
      a.row_stat[static_cast<size_t>(b) * a.Hq + a.heads[g * G + h]] = make_float2(M * kLn2, inv);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int h = e / D, dd = e % D;
    const int hq = a.heads[g * G + h];
    const float* pp = a.part + (static_cast<size_t>(b) * a.Hq + hq) * a.S * (D + 4);
    float acc = 0.f;
#pragma unroll 4
    for (int s = 0; s < a.S; ++s) acc += wts[h * a.S + s] * __ldcg(pp + s * (D + 4) + 4 + dd);
    static_cast<__nv_bfloat16*>(a.out)[(static_cast<size_t>(b) * a.Hq + hq) * D + dd] =
        __float2bfloat16_rn(acc);
  }
  if (threadIdx.x == 0) a.counters[unit] = 0u;   // ready for the next launch
}

// ------------------------------------------------------------------------
// Dense / anchor decode, TMA producer warp + NW consumer warps.
// ------------------------------------------------------------------------
// Fused anchor decode: the lanes of one head (those with the same c4) file
// the logits of their keys whose order-preserving key is >= t_lo in the
// warp's own sub-list of the row, at positions from a ballot prefix.
__device__ __forceinline__ void filter_file(bool in, uint32_t key, int pos, uint32_t group,
                                            uint32_t below, uint2* list, uint32_t& cnt) {
  const uint32_t bits = __ballot_sync(0xffffffffu, in) & group;
  if (in) list[cnt + __popc(bits & below)] = make_uint2(key, static_cast<uint32_t>(pos));
  cnt += __popc(bits);
}

template <int D, int NW, int STAGES, bool SPILL, bool FILTER>
__global__ void __launch_bounds__((NW + 1) * 32)
    k_decode_dense_bf16(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ DecodeArgs a) {
  pdl_wait();
  pdl_trigger();
  constexpr int TK = 16 * NW;
  constexpr int HALVES = D / 64;
  constexpr int TILE_BYTES = HALVES * TK * 128;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* ktile = smem;
  unsigned char* vtile = smem + STAGES * TILE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(vtile + STAGES * TILE_BYTES);
  uint64_t* empty = full + STAGES;

  const int split = blockIdx.x, unit = blockIdx.y;
  const int b = unit / a.Hkv, g = unit % a.Hkv;
  const int n0 = split * a.chunk;
  const int n1 = min(a.N, n0 + a.chunk);
  const int ntiles = n0 < n1 ? (n1 - n0 + TK - 1) / TK : 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    fence_barrier_init();
  }
  __syncthreads();

  WarpState<D> st;
  warp_state_init(st);
  if (warp == NW) {
    // ---------------- producer ----------------
    if (lane == 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const int row_base = unit * a.N + n0;
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % STAGES;
        if (!mbar_wait(&empty[s], ((t / STAGES) & 1) ^ 1, a.err, 0x101)) break;
        mbar_arrive_expect_tx(&full[s], 2 * TILE_BYTES);
#pragma unroll
        for (int hf = 0; hf < HALVES; ++hf) {
          tma_load_2d(ktile + s * TILE_BYTES + hf * TK * 128, &tmK, &full[s], hf * 64,
                      row_base + t * TK);
          tma_load_2d(vtile + s * TILE_BYTES + hf * TK * 128, &tmV, &full[s], hf * 64,
                      row_base + t * TK);
        }
        issued = t + 1;
      }
      // Never leave with copies in flight.
      for (int t = issued > STAGES ? issued - STAGES : 0; t < issued; ++t)
        mbar_wait(&full[t % STAGES], (t / STAGES) & 1, a.err, 0x102);
    }
  } else {
    // ---------------- consumers ----------------
    uint32_t qf[D / 16][2];
    load_q_frags<D>(a, b, g, qf);
    const int gid = lane >> 2, c4 = lane & 3;
    const int row0 = warp * 16;
    const bool hv0 = 2 * c4 < a.G, hv1 = 2 * c4 + 1 < a.G;
    float* sp0 = nullptr;
    float* sp1 = nullptr;
    const int row_h0 = hv0 ? b * a.Hq + a.heads[g * a.G + 2 * c4] : 0;
    const int row_h1 = hv1 ? b * a.Hq + a.heads[g * a.G + 2 * c4 + 1] : 0;
    if (SPILL) {
      if (hv0) sp0 = a.spill + static_cast<size_t>(row_h0) * a.N;
      if (hv1) sp1 = a.spill + static_cast<size_t>(row_h1) * a.N;
    }
    uint32_t tlo0 = 0xFFFFFFFFu, tlo1 = 0xFFFFFFFFu;
    uint2* fl0 = nullptr;
    uint2* fl1 = nullptr;
    uint32_t fc0 = 0, fc1 = 0;
    const uint32_t fgroup = 0x11111111u << c4;                 // lanes of this head pair
    const uint32_t fbelow = fgroup & ((1u << lane) - 1u);
    const int fsub = (NW > 0) ? a.chunk / NW : 0;               // sub-list capacity
    if (FILTER) {
      const size_t sub = static_cast<size_t>(split) * a.chunk + static_cast<size_t>(warp) * fsub;
      if (hv0) {
        tlo0 = a.bracket[row_h0].x;
        fl0 = a.flist + static_cast<size_t>(row_h0) * a.S * a.chunk + sub;
      }
      if (hv1) {
        tlo1 = a.bracket[row_h1].x;
        fl1 = a.flist + static_cast<size_t>(row_h1) * a.S * a.chunk + sub;
      }
    }
    bool fbad = false;
    for (int t = 0; t < ntiles; ++t) {
      const int s = t % STAGES;
      if (!mbar_wait_warp(&full[s], (t / STAGES) & 1, a.err, 0x103)) break;
      float sc[4];
      slice_scores<D>(smem_u32(ktile + s * TILE_BYTES), TK, row0, qf, sc);
      const int key0 = n0 + t * TK + row0 + gid, key1 = key0 + 8;
      const bool kv0 = key0 < n1, kv1 = key1 < n1;
      if (SPILL) {
        const float v0 = sc[0] * a.scale, v1 = sc[1] * a.scale;
        const float v2 = sc[2] * a.scale, v3 = sc[3] * a.scale;
        if (kv0) {
          if (hv0) sp0[key0] = v0;
          if (hv1) sp1[key0] = v1;
        }
        if (kv1) {
          if (hv0) sp0[key1] = v2;
          if (hv1) sp1[key1] = v3;
        }
        if (FILTER) {
          // the same fp32 values the spill holds, so the selection made from
          // the lists equals the one made from the spill
          fbad |= (kv0 && ((hv0 && v0 != v0) || (hv1 && v1 != v1))) ||
                  (kv1 && ((hv0 && v2 != v2) || (hv1 && v3 != v3)));
          const uint32_t f0 = float_key_fast(v0), f1 = float_key_fast(v1);
          const uint32_t f2 = float_key_fast(v2), f3 = float_key_fast(v3);
          filter_file(kv0 && hv0 && f0 >= tlo0, f0, key0, fgroup, fbelow, fl0, fc0);
          filter_file(kv1 && hv0 && f2 >= tlo0, f2, key1, fgroup, fbelow, fl0, fc0);
          filter_file(kv0 && hv1 && f1 >= tlo1, f1, key0, fgroup, fbelow, fl1, fc1);
          filter_file(kv1 && hv1 && f3 >= tlo1, f3, key1, fgroup, fbelow, fl1, fc1);
        }
      }
      float x[4];
      x[0] = kv0 ? sc[0] * a.scale_log2 : kNegInf;
      x[1] = kv0 ? sc[1] * a.scale_log2 : kNegInf;
      x[2] = kv1 ? sc[2] * a.scale_log2 : kNegInf;
      x[3] = kv1 ? sc[3] * a.scale_log2 : kNegInf;
      slice_softmax_pv<D>(st, x, smem_u32(vtile + s * TILE_BYTES), TK, row0);
      // The stage is refilled by TMA (the async proxy) once every consumer
      // warp has released it; the mbarrier alone did not order this warp's
      // ldmatrix reads (generic proxy) before that write: without the fence
      // a refill occasionally overwrote the last V columns still being read
      // (about one long-shape anchor layer in sixteen came out wrong).
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (FILTER) {
      // a NaN logit: the selection from the lists would not see it
      if (__any_sync(0xffffffffu, fbad) && lane == 0)
        report_error(a.err, KASCADE_ERR_BAD_INPUT, 0x104);
      // sub-list lengths, one writer per (row, split, warp)
      if (gid == 0) {
        if (hv0) a.fcount[(static_cast<size_t>(row_h0) * a.S + split) * NW + warp] = fc0;
        if (hv1) a.fcount[(static_cast<size_t>(row_h1) * a.S + split) * NW + warp] = fc1;
      }
    }
  }
  __syncthreads();
  finish_cta<D>(a, st, warp < NW ? warp : -1, NW, reinterpret_cast<float*>(smem), b, g, split);
}

// ------------------------------------------------------------------------
// Union plan, one CTA per (key-range chunk c, sequence b, KV head g): the G
// ascending per-head sets are cut to keys [c*R, (c+1)*R) by a warp-wide
// 32-ary lower-bound search, marked in per-slot shared bitmaps and emitted as
// one ascending list of entries key | (head-slot mask << 24) into
// plan[unit][c][kPlanCap], with its length in plan_count[unit][c]. Reuse
// CTA (c, unit) consumes exactly chunk c.
// ------------------------------------------------------------------------
__device__ __forceinline__ int warp_lower_bound(const int32_t* row, int n, int v) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = n;   // first index in [lo, hi] with row[i] >= v
  while (hi - lo > 32) {
    const int step = (hi - lo + 31) / 32;
    const int p = lo + (lane + 1) * step - 1;
    const bool ge = p >= hi || __ldg(row + p) >= v;
    const unsigned int bal = __ballot_sync(0xffffffffu, ge);
    if (bal == 0u) return hi;
    const int f = __ffs(bal) - 1;
    const int nlo = f == 0 ? lo : lo + f * step;
    hi = min(hi, lo + (f + 1) * step - 1);
    lo = nlo;
  }
  const int p = lo + lane;
  const bool ge = p < hi && __ldg(row + p) >= v;
  const unsigned int bal = __ballot_sync(0xffffffffu, ge);
  return bal ? lo + __ffs(bal) - 1 : hi;
}

__global__ void __launch_bounds__(256) k_build_union_plan(const __grid_constant__ DecodeArgs a,
                                                          uint32_t* __restrict__ plan,
                                                          int32_t* __restrict__ plan_count,
                                                          int R) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t bm[8][kPlanCap / 32];
  __shared__ int s_lo[8], s_hi[8];
  __shared__ int s_scan[256];
  const int c = blockIdx.x, unit = blockIdx.y, nch = gridDim.x;
  const int b = unit / a.Hkv, g = unit % a.Hkv;
  const int G = a.G, topk = a.topk;
  const int n0 = c * R, n1 = min(a.N, n0 + R);
  const int words = (R + 31) / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // sets of this unit: one per query head of the group, or the group's one
  // pooled set (whose entries then carry every head of the group)
  const int nsets = a.pooled ? 1 : G;
  auto set_row = [&](int slot) {
    return a.pooled ? a.idx + static_cast<size_t>(unit) * topk
                    : a.idx + (static_cast<size_t>(b) * a.Hq + a.heads[g * G + slot]) * topk;
  };
  for (int i = threadIdx.x; i < nsets * words; i += blockDim.x) bm[i / words][i % words] = 0u;
  // search job j: the chunk start of set j (j < nsets) or the chunk end of
  // set j - nsets, spread over the 8 warps so the searches run concurrently
  for (int job = warp; job < 2 * nsets; job += 8) {
    const int slot = job < nsets ? job : job - nsets;
    const bool is_hi = job >= nsets;
    const int32_t* row = set_row(slot);
    const int pos = warp_lower_bound(row, topk, is_hi ? n1 : n0);
    if (lane == 0) {
      if (is_hi) s_hi[slot] = pos;
      else s_lo[slot] = pos;
      // entries below 0 (first chunk) or at/after N (last chunk) are invalid
      if ((!is_hi && c == 0 && pos > 0) || (is_hi && c == nch - 1 && pos < topk))
        report_error(a.err, KASCADE_ERR_BAD_INPUT, 0x201);
    }
  }
  __syncthreads();
  for (int slot = 0; slot < nsets; ++slot) {
    const int32_t* row = set_row(slot);
    const int hi = s_hi[slot];
    for (int i = s_lo[slot] + threadIdx.x; i < hi; i += blockDim.x) {
      const int raw = __ldg(row + i);
      const int key = raw - n0;
      // the sets must be strictly ascending and inside [0, N)
      if (key < 0 || key >= n1 - n0 || (i + 1 < hi && __ldg(row + i + 1) <= raw)) {
        report_error(a.err, KASCADE_ERR_BAD_INPUT, 0x202);
        if (key < 0 || key >= n1 - n0) continue;
      }
      atomicOr(&bm[slot][key >> 5], 1u << (key & 31));
    }
  }
  __syncthreads();
  // contiguous word runs per thread; block scan of union counts
  const int per = (words + blockDim.x - 1) / blockDim.x;
  const int w0 = min(words, static_cast<int>(threadIdx.x) * per), w1 = min(words, w0 + per);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) {
    uint32_t u = 0;
    for (int slot = 0; slot < nsets; ++slot) u |= bm[slot][w];
    cnt += __popc(u);
  }
  s_scan[threadIdx.x] = cnt;
  __syncthreads();
  for (int off = 1; off < static_cast<int>(blockDim.x); off <<= 1) {
    const int v = static_cast<int>(threadIdx.x) >= off ? s_scan[threadIdx.x - off] : 0;
    __syncthreads();
    s_scan[threadIdx.x] += v;
    __syncthreads();
  }
  int pos = s_scan[threadIdx.x] - cnt;
  uint32_t* out = plan + (static_cast<size_t>(unit) * nch + c) * kPlanCap;
  for (int w = w0; w < w1; ++w) {
    uint32_t u = 0;
    for (int slot = 0; slot < nsets; ++slot) u |= bm[slot][w];
    while (u) {
      const int bit = __ffs(u) - 1;
      u &= u - 1;
      uint32_t mask = a.pooled ? (1u << G) - 1u : 0u;
      if (!a.pooled)
        for (int slot = 0; slot < G; ++slot) mask |= ((bm[slot][w] >> bit) & 1u) << slot;
      out[pos++] = static_cast<uint32_t>(n0 + w * 32 + bit) | (mask << 24);
    }
  }
  if (threadIdx.x == blockDim.x - 1) plan_count[unit * nch + c] = s_scan[threadIdx.x];
}

// The same plan from the heads' selection bitmaps (one word per 32 keys per
// query-head row, as the anchor layer's Top-k emits them): CTA (c, unit)
// ORs the G rows' words of keys [c*R, (c+1)*R) and emits the union in key
// order with each entry's head mask, exactly as k_build_union_plan does from
// the sets, without searching them. Per-head sets only.
__global__ void __launch_bounds__(256) k_build_union_plan_bits(const __grid_constant__ DecodeArgs a,
                                                               const uint32_t* __restrict__ sel,
                                                               int words_per_row,
                                                               uint32_t* __restrict__ plan,
                                                               int32_t* __restrict__ plan_count,
                                                               int R) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_scan[256];
  const int c = blockIdx.x, unit = blockIdx.y, nch = gridDim.x;
  const int b = unit / a.Hkv, g = unit % a.Hkv;
  const int G = a.G;
  const int n0 = c * R, n1 = min(a.N, n0 + R);
  const int words = (n1 - n0 + 31) / 32;   // R is a multiple of 32
  const int w_base = n0 / 32;
  // contiguous word runs per thread (at most one word for R <= 8192)
  const int per = (words + blockDim.x - 1) / blockDim.x;
  const int w0 = min(words, static_cast<int>(threadIdx.x) * per), w1 = min(words, w0 + per);
  auto word_of = [&](int slot, int w) {
    const size_t row = static_cast<size_t>(b) * a.Hq + a.heads[g * G + slot];
    return __ldg(sel + row * words_per_row + w_base + w);
  };
  int cnt = 0;
  for (int w = w0; w < w1; ++w) {
    uint32_t u = 0;
    for (int slot = 0; slot < G; ++slot) u |= word_of(slot, w);
    cnt += __popc(u);
  }
  s_scan[threadIdx.x] = cnt;
  __syncthreads();
  for (int off = 1; off < static_cast<int>(blockDim.x); off <<= 1) {
    const int v = static_cast<int>(threadIdx.x) >= off ? s_scan[threadIdx.x - off] : 0;
    __syncthreads();
    s_scan[threadIdx.x] += v;
    __syncthreads();
  }
  int pos = s_scan[threadIdx.x] - cnt;
  uint32_t* out = plan + (static_cast<size_t>(unit) * nch + c) * kPlanCap;
  for (int w = w0; w < w1; ++w) {
    uint32_t bw[8];
    uint32_t u = 0;
    for (int slot = 0; slot < G; ++slot) {
      bw[slot] = word_of(slot, w);
      u |= bw[slot];
    }
    while (u) {
      const int bit = __ffs(u) - 1;
      u &= u - 1;
      uint32_t mask = 0u;
      for (int slot = 0; slot < G; ++slot) mask |= ((bw[slot] >> bit) & 1u) << slot;
      out[pos++] = static_cast<uint32_t>(n0 + w * 32 + bit) | (mask << 24);
    }
  }
  if (threadIdx.x == blockDim.x - 1) plan_count[unit * nch + c] = s_scan[threadIdx.x];
}

// ------------------------------------------------------------------------
// Reuse decode over the union plan. A CTA takes an equal run of the 16-row
// slices of one (sequence, KV head), numbered across the unit's plan chunks
// in key order, as one stream; every warp gathers its own slices through a
// STAGES-deep cp.async pipeline (no block barriers), reading each slice's
// plan entries from global memory one slice ahead. Padding entries (mask 0)
// are zero-filled, never read.
// ------------------------------------------------------------------------

// DIRECT (pooled index sets): every head of a group shares the group's one
// ascending set, so the set itself is the gather list, with every head's bit
// in the mask, and no plan is built; a.S CTAs per (sequence, KV head) take
// equal runs of its 16-row slices. Entries outside [0, N) or out of order
// are reported as bad input and not read.
template <int D, int NW, int STAGES, bool DIRECT>
__global__ void __launch_bounds__(NW * 32)
    k_decode_union_bf16(const __grid_constant__ DecodeArgs a) {
  pdl_wait();
  pdl_trigger();
  constexpr int SLICE = (D / 64) * 16 * 128;     // bytes of one K (or V) slice
  constexpr int CHUNKS = D / 8;                   // 16-byte chunks per row
  constexpr int ROWS_PER_INSTR = 32 / CHUNKS;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ int s_pref[kMaxSplits + 1];                // slice prefix over the unit's chunks
  __shared__ int s_cnt[kMaxSplits];                     // plan entries of the unit's chunks
  __shared__ uint32_t s_ent[NW][STAGES][16];            // entries of the slices in flight
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* wbuf = smem + warp * STAGES * 2 * SLICE;

  const int split = blockIdx.x, unit = blockIdx.y;
  const int b = unit / a.Hkv, g = unit % a.Hkv;
  // The unit's 16-row slices, numbered across its plan chunks in key order
  // (DIRECT: across its set), are split into a.S equal runs, one per CTA, so
  // no CTA waits on a longer one of the same unit.
  const int nch = DIRECT ? 0 : a.plan_chunks;
  if (!DIRECT && warp == 0) {
    // every chunk's entry count, 32 chunks per round, and a running prefix
    int carry = 0;
    for (int cb = 0; cb < nch; cb += 32) {
      const int c = cb + lane;
      const int cnt = c < nch ? min(kPlanCap, a.plan_count[unit * nch + c]) : 0;
      const int sl = (cnt + 15) / 16;
      int incl = sl;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (c < nch) {
        s_cnt[c] = cnt;
        s_pref[c] = carry + incl - sl;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_pref[nch] = carry;
  }
  __syncthreads();
  const int total = DIRECT ? (a.topk + 15) / 16 : s_pref[nch];
  const int per = (total + a.S - 1) / a.S;
  const int g0 = min(total, split * per);
  const int nslices = min(total, g0 + per) - g0;
  const int my = warp < nslices ? (nslices - warp + NW - 1) / NW : 0;
  const int32_t* dset = DIRECT ? a.idx + static_cast<size_t>(unit) * a.topk : nullptr;
  const uint32_t dmask = (1u << a.G) - 1u;
  int fc = 0;   // chunk cursor: a warp's slices only move forward
  // this lane's plan entry of slice sl of the CTA (lanes 16..31 repeat 0..15)
  auto fetch = [&](int sl) -> uint32_t {
    const int gs = g0 + sl;
    while (fc + 1 < nch && s_pref[fc + 1] <= gs) ++fc;
    const int e = (gs - s_pref[fc]) * 16 + (lane & 15);
    return e < s_cnt[fc] ? __ldg(a.plan + (static_cast<size_t>(unit) * nch + fc) * kPlanCap + e)
                         : 0u;
  };
  // DIRECT: this lane's set entry of slice sl and the entry before it, loaded
  // here but checked (direct_entry) only when the slice's copies are issued a
  // slice later; checking right after the loads stalled every warp a whole
  // load latency per slice (pooled 8B decode shape: 34 us, DRAM half busy)
  auto fetch_direct = [&](int sl) -> int2 {
    const int e = (g0 + sl) * 16 + (lane & 15);
    if (e >= a.topk) return make_int2(0, 0);
    return make_int2(__ldg(dset + e), e > 0 ? __ldg(dset + e - 1) : -1);
  };
  auto direct_entry = [&](int sl, int2 r) -> uint32_t {
    const int e = (g0 + sl) * 16 + (lane & 15);
    if (e >= a.topk) return 0u;   // past the set: padding
    if (r.x < 0 || r.x >= a.N || r.x <= r.y) {
      report_error(a.err, KASCADE_ERR_BAD_INPUT, 0x203);
      return 0u;   // padding: not read
    }
    return static_cast<uint32_t>(r.x) | (dmask << 24);
  };
  const __nv_bfloat16* kbase =
      static_cast<const __nv_bfloat16*>(a.k) + static_cast<size_t>(unit) * a.N * D;
  const __nv_bfloat16* vbase =
      static_cast<const __nv_bfloat16*>(a.v) + static_cast<size_t>(unit) * a.N * D;

  // Per-head sets: slice i's K rows go to K buffer i % STAGES and its V rows
  // to V buffer i % STAGES, each as its own cp.async group. A K buffer is free
  // once the scores of its slice are formed and a V buffer once its P V
  // product is, so slice i + STAGES's K copies start in the middle of slice
  // i's work and its V copies at the end: STAGES slices stay in flight per
  // warp (8B decode shape: 81.7 -> 80.6 us per reuse layer).
  auto issue_half = [&](int i, uint32_t ent, bool is_v) {
    const int stg = i % STAGES;
    if (!is_v && lane < 16) s_ent[warp][stg][lane] = ent;
    unsigned char* dst = wbuf + stg * 2 * SLICE + (is_v ? SLICE : 0);
    const __nv_bfloat16* src = is_v ? vbase : kbase;
#pragma unroll
    for (int it = 0; it < 16 / ROWS_PER_INSTR; ++it) {
      const int row = it * ROWS_PER_INSTR + lane / CHUNKS;
      const int ch = lane % CHUNKS;
      const uint32_t ent_r = __shfl_sync(0xffffffffu, ent, row);
      const bool ok = (ent_r >> 24) != 0u;   // padding: mask 0
      const size_t off = static_cast<size_t>(ent_r & 0xFFFFFFu) * D + ch * 8;
      cp_async16(dst + sw128_offset(16, row, ch), src + off, ok ? 16u : 0u);
    }
  };

  WarpState<D> st;
  warp_state_init(st);
  uint32_t qf[D / 16][2];
  load_q_frags<D>(a, b, g, qf);
  const int gid = lane >> 2, c4 = lane & 3;

  if constexpr (!DIRECT) {
  #pragma unroll
    for (int i = 0; i < STAGES; ++i) {
      const uint32_t e = i < my ? fetch(warp + i * NW) : 0u;
      if (i < my) issue_half(i, e, false);
      cp_async_commit();
      if (i < my) issue_half(i, e, true);
      cp_async_commit();
    }
    // entries of the next slice to issue, read one iteration before its copies
    uint32_t nxt = STAGES < my ? fetch(warp + STAGES * NW) : 0u;
    for (int i = 0; i < my; ++i) {
      // slice i's K and V groups have landed once at most the 2 (STAGES - 1)
      // groups issued after them are pending
      cp_async_wait<2 * (STAGES - 1)>();
      __syncwarp();
      const int stg = i % STAGES;
      const uint32_t kd = smem_u32(wbuf + stg * 2 * SLICE);
      float sc[4];
      slice_scores<D>(kd, 16, 0, qf, sc);
      const uint32_t ent = s_ent[warp][stg][lane & 15];
      const uint32_t m0 = __shfl_sync(0xffffffffu, ent, gid) >> 24;
      const uint32_t m1 = __shfl_sync(0xffffffffu, ent, gid + 8) >> 24;
      // the K buffer and this stage's entries are free: slice i + STAGES's K
      const int nx = i + STAGES;
      const uint32_t ent_n = nxt;
      nxt = nx + 1 < my ? fetch(warp + (nx + 1) * NW) : 0u;
      __syncwarp();
      if (nx < my) issue_half(nx, ent_n, false);
      cp_async_commit();
      float x[4];
      x[0] = ((m0 >> (2 * c4)) & 1u) ? sc[0] * a.scale_log2 : kNegInf;
      x[1] = ((m0 >> (2 * c4 + 1)) & 1u) ? sc[1] * a.scale_log2 : kNegInf;
      x[2] = ((m1 >> (2 * c4)) & 1u) ? sc[2] * a.scale_log2 : kNegInf;
      x[3] = ((m1 >> (2 * c4 + 1)) & 1u) ? sc[3] * a.scale_log2 : kNegInf;
      slice_softmax_pv<D>(st, x, kd + SLICE, 16, 0);
      // the V buffer is free: slice i + STAGES's V
      __syncwarp();
      if (nx < my) issue_half(nx, ent_n, true);
      cp_async_commit();
    }
  } else {
    // pooled sets: slice i + STAGES - 1 (K and V together) is requested at the
    // top of iteration i into the buffers slice i - 1 used (measured faster
    // here than the split requests: 35.5 against 37.0 us per pooled layer)
    int2 raw = my > 0 ? fetch_direct(warp) : make_int2(0, 0);
#pragma unroll
    for (int i = 0; i < STAGES - 1; ++i) {
      if (i < my) {
        const uint32_t e = direct_entry(warp + i * NW, raw);
        raw = (i + 1 < my) ? fetch_direct(warp + (i + 1) * NW) : make_int2(0, 0);
        issue_half(i, e, false);
        issue_half(i, e, true);
      }
      cp_async_commit();
    }
    for (int i = 0; i < my; ++i) {
      if (i + STAGES - 1 < my) {
        const uint32_t e = direct_entry(warp + (i + STAGES - 1) * NW, raw);
        raw = (i + STAGES < my) ? fetch_direct(warp + (i + STAGES) * NW) : make_int2(0, 0);
        issue_half(i + STAGES - 1, e, false);
        issue_half(i + STAGES - 1, e, true);
      }
      cp_async_commit();
      cp_async_wait<STAGES - 1>();
      __syncwarp();
      const uint32_t kd = smem_u32(wbuf + (i % STAGES) * 2 * SLICE);
      float sc[4];
      slice_scores<D>(kd, 16, 0, qf, sc);
      const uint32_t ent = s_ent[warp][i % STAGES][lane & 15];
      const uint32_t m0 = __shfl_sync(0xffffffffu, ent, gid) >> 24;
      const uint32_t m1 = __shfl_sync(0xffffffffu, ent, gid + 8) >> 24;
      float x[4];
      x[0] = ((m0 >> (2 * c4)) & 1u) ? sc[0] * a.scale_log2 : kNegInf;
      x[1] = ((m0 >> (2 * c4 + 1)) & 1u) ? sc[1] * a.scale_log2 : kNegInf;
      x[2] = ((m1 >> (2 * c4)) & 1u) ? sc[2] * a.scale_log2 : kNegInf;
      x[3] = ((m1 >> (2 * c4 + 1)) & 1u) ? sc[3] * a.scale_log2 : kNegInf;
      slice_softmax_pv<D>(st, x, kd + SLICE, 16, 0);
      __syncwarp();
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  finish_cta<D>(a, st, warp, NW, reinterpret_cast<float*>(smem), b, g, split);
}

// ------------------------------------------------------------------------
// Generic CUDA-core decode: one CTA per (query head, sequence); fp32 inputs.
// Logits go to the spill buffer (always present on this path), then a block
// softmax and a dim-parallel weighted sum of V.
// ------------------------------------------------------------------------
__device__ float block_reduce(float v, bool is_max, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int off = 16; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  float r = is_max ? kNegInf : 0.f;
  for (int w = 0; w < nw; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
  return r;
}

__global__ void k_decode_generic_f32(const __grid_constant__ DecodeArgs a, int D, int kind) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float qs[];   // [D]
  __shared__ float red[32];
  const int b = blockIdx.y, hq = blockIdx.x;
  int g = 0;
  for (int gg = 0; gg < a.Hkv; ++gg)
    for (int s = 0; s < a.G; ++s)
      if (a.heads[gg * a.G + s] == hq) g = gg;
  const float* q = static_cast<const float*>(a.q) + (static_cast<size_t>(b) * a.Hq + hq) * D;
  const float* K = static_cast<const float*>(a.k) + (static_cast<size_t>(b) * a.Hkv + g) * a.N * D;
  const float* V = static_cast<const float*>(a.v) + (static_cast<size_t>(b) * a.Hkv + g) * a.N * D;
  float* s = a.spill + (static_cast<size_t>(b) * a.Hq + hq) * a.N;
  const int32_t* sel =
      (kind == kSparse)
          ? a.idx + (a.pooled ? static_cast<size_t>(b) * a.Hkv + g
                              : static_cast<size_t>(b) * a.Hq + hq) * a.topk
          : nullptr;
  const int n = (kind == kSparse) ? a.topk : a.N;
  for (int c = threadIdx.x; c < D; c += blockDim.x) qs[c] = q[c];
  __syncthreads();
  float mx = kNegInf;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    int key = j;
    if (sel) {
      key = sel[j];
      if (key < 0 || key >= a.N) {
        report_error(a.err, KASCADE_ERR_BAD_INPUT, 0x301);
        key = 0;
      }
    }
    float acc = 0.f;
    for (int c = 0; c < D; ++c) acc = fmaf(qs[c], K[static_cast<size_t>(key) * D + c], acc);
    acc *= a.scale;
    s[j] = acc;              // sparse: slot j of the set; dense: key j
    mx = fmaxf(mx, acc);
  }
  mx = block_reduce(mx, true, red);
  float sum = 0.f;
  for (int j = threadIdx.x; j < n; j += blockDim.x) sum += expf(s[j] - mx);
  sum = block_reduce(sum, false, red);
  const float inv = 1.f / sum;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < n; ++j) {
      int key = sel ? sel[j] : j;
      if (key < 0 || key >= a.N) key = 0;
      acc = fmaf(expf(s[j] - mx), V[static_cast<size_t>(key) * D + c], acc);
    }
    static_cast<float*>(a.out)[(static_cast<size_t>(b) * a.Hq + hq) * D + c] = acc * inv;
  }
}

template <int D, int NW, int STAGES, bool SPILL, bool FILTER>
cudaError_t launch_dense_t(const DecodeArgs& a, cudaStream_t st) {
  constexpr int TK = 16 * NW;
  alignas(64) CUtensorMap tk, tv;
  const uint64_t rows = static_cast<uint64_t>(a.B) * a.Hkv * a.N;
  if (!encode_tmap_2d_bf16(&tk, a.k, D, rows, 64, TK, true)) return cudaErrorInvalidValue;
  if (!encode_tmap_2d_bf16(&tv, a.v, D, rows, 64, TK, true)) return cudaErrorInvalidValue;
  constexpr int TILE_BYTES = (D / 64) * TK * 128;
  const size_t smem = 1024 + 2 * STAGES * TILE_BYTES + 2 * STAGES * 8;
  auto kern = k_decode_dense_bf16<D, NW, STAGES, SPILL, FILTER>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(a.S, a.B * a.Hkv);
  return launch_pdl(kern, grid, dim3((NW + 1) * 32), smem, st, tk, tv, a);
}

template <int D, int NW, int STAGES, bool DIRECT>
cudaError_t launch_union_t(const DecodeArgs& a, cudaStream_t st) {
  constexpr int SLICE = (D / 64) * 16 * 128;
  const size_t smem = 1024 + static_cast<size_t>(NW) * STAGES * 2 * SLICE;
  auto kern = k_decode_union_bf16<D, NW, STAGES, DIRECT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // resident CTAs of this kernel (queried once per device)
  // per host thread, so concurrent callers never race on the cache
  thread_local int cached_dev = -1, cached_slots = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidValue;
  if (dev != cached_dev) {
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, smem) != cudaSuccess)
      return cudaErrorInvalidValue;
    cached_slots = max(1, sms * per_sm);
    cached_dev = dev;
  }
  // equal runs of each unit's slices, as many CTAs per unit as fill one
  // wave of resident CTAs (a second, partial wave costs more than slots left
  // idle); a.S is the unit's plan chunks (unused with DIRECT)
  DecodeArgs u = a;
  const int units = a.B * a.Hkv;
  const int max_slices = DIRECT ? (a.topk + 15) / 16 : a.S * (kPlanCap / 16);
  u.plan_chunks = DIRECT ? 0 : a.S;
  u.chunks_per_cta = 0;
  u.S = max(1, min(cached_slots / units, min(max_slices, kMaxSplits)));
  dim3 grid(u.S, a.B * a.Hkv);
  return launch_pdl(kern, grid, dim3(NW * 32), smem, st, u);
}

}  // namespace

// Launch shapes: 4 consumer warps (64-key tiles) per CTA. Dense decode runs
// 152 * 8 split CTAs (three resident per SM, so about 2.7 waves; 152 * 6 and
// 152 * 12 were both slower); the union gather sizes its CTAs to one wave.
constexpr int kDenseNW = kDecodeConsumerWarps;
constexpr int kUnionNW = 4;
constexpr int kTargetCtas = 152 * 2 * 4;
constexpr int kUnionTargetCtas = 152 * 2 * 4;

int decode_chunk_dense(int units, int N) {
  int s = (kTargetCtas + units - 1) / units;
  if (s < 1) s = 1;
  int chunk = (N + s - 1) / s;
  const int min_chunk = (N + kMaxSplits - 1) / kMaxSplits;
  if (chunk < min_chunk) chunk = min_chunk;
  if (chunk < 256) chunk = 256;
  return (chunk + 63) & ~63;
}

// Key-range chunks of the reuse decode: R keys (multiple of 32, at most
// kPlanCap so a chunk's union fits the shared staging area), about four
// waves of CTAs over 152 SMs x 2, and at most kMaxSplits chunks per (sequence,
// KV head) (the split merge holds that many partials): few units on long
// rows take longer chunks, up to N = kMaxSplits * kPlanCap.
int decode_union_range(int units, int N) {
  int s = (kUnionTargetCtas + units - 1) / units;
  if (s < 1) s = 1;
  int R = (N + s - 1) / s;
  R = (R + 31) & ~31;
  if (R < 256) R = 256;
  const int r_min = ((N + kMaxSplits - 1) / kMaxSplits + 31) & ~31;
  if (R < r_min) R = r_min;
  if (R > kPlanCap) R = kPlanCap;
  return R;
}
int decode_union_chunks(int units, int N) {
  const int R = decode_union_range(units, N);
  return (N + R - 1) / R;
}

cudaError_t launch_decode_dense_bf16(const DecodeArgs& a, int head_dim, bool spill,
                                     cudaStream_t st, bool filter) {
  if (filter && !spill) return cudaErrorInvalidValue;
  if (head_dim == 128)
    // two 32 KB stages: 64 KB, three CTAs per SM (three stages at two per SM
    // were 2% slower)
    return filter  ? launch_dense_t<128, kDenseNW, 2, true, true>(a, st)
           : spill ? launch_dense_t<128, kDenseNW, 2, true, false>(a, st)
                   : launch_dense_t<128, kDenseNW, 2, false, false>(a, st);
  if (head_dim == 64)
    // four 16 KB stages: 64 KB, three CTAs per SM (six stages, two per SM, were
    // 4% slower on 131072-key rows)
    return filter  ? launch_dense_t<64, kDenseNW, 4, true, true>(a, st)
           : spill ? launch_dense_t<64, kDenseNW, 4, true, false>(a, st)
                   : launch_dense_t<64, kDenseNW, 4, false, false>(a, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_union_bf16(const DecodeArgs& a, int head_dim, cudaStream_t st) {
  // pooled sets carry k rows per unit instead of the ~G k / 2 of a union, so
  // their CTAs are shorter: one more stage in flight per warp pays there;
  // they are gathered straight from the sets (no plan)
  if (head_dim == 128)
    // (per-head sets: three stages at two CTAs per SM measured 82.4 against
    // 81.8 us for two at three per SM on the 8B decode shape)
    return a.pooled ? launch_union_t<128, kUnionNW, 3, true>(a, st)
                    : launch_union_t<128, kUnionNW, 2, false>(a, st);
  if (head_dim == 64)
    // (per-head sets, 131072-key rows: four 16 KB stages at three CTAs per SM
    // 116.7 us against 123.7 / 131 / 125 us for two / three / six stages on
    // rotating layers; 89.1 against 90.6 us per reuse layer in the long stack)
    return a.pooled ? launch_union_t<64, kUnionNW, 3, true>(a, st)
                    : launch_union_t<64, kUnionNW, 4, false>(a, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_build_union_plan_bits(const DecodeArgs& a, const uint32_t* sel, int words,
                                         uint32_t* plan, int32_t* plan_count, cudaStream_t st) {
  if (a.G > 8 || a.pooled) return cudaErrorInvalidValue;
  const int R = decode_union_range(a.B * a.Hkv, a.N);
  const int S = (a.N + R - 1) / R;
  if (S > kMaxSplits) return cudaErrorNotSupported;
  return launch_pdl(k_build_union_plan_bits, dim3(S, a.B * a.Hkv), dim3(256), 0, st, a, sel,
                    words, plan, plan_count, R);
}

cudaError_t launch_build_union_plan(const DecodeArgs& a, uint32_t* plan, int32_t* plan_count,
                                    cudaStream_t st) {
  if (a.G > 8) return cudaErrorInvalidValue;
  const int R = decode_union_range(a.B * a.Hkv, a.N);
  const int S = (a.N + R - 1) / R;
  if (S > kMaxSplits) return cudaErrorNotSupported;
  return launch_pdl(k_build_union_plan, dim3(S, a.B * a.Hkv), dim3(256), 0, st, a, plan,
                    plan_count, R);
}

cudaError_t launch_decode_generic(const DecodeArgs& a, int head_dim, int dtype, DecodeKind kind,
                                  cudaStream_t st) {
  if (dtype != KASCADE_F32) return cudaErrorInvalidValue;
  dim3 grid(a.Hq, a.B);
  return launch_pdl(k_decode_generic_f32, grid, dim3(256), head_dim * sizeof(float), st, a,
                    head_dim, static_cast<int>(kind));
}

}  // namespace kascade
