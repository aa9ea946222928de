// api.cu — the C ABI of libkascade (include/kascade.h): argument validation,
// workspace layout, kernel dispatch and the layer-stack driver.
//
// Stack semantics follow the Kascade pages (euno.news summary, Key
// Contributions "Cross-layer Top-k reuse", Methodology 2-3): an anchor layer
// computes exact attention and replaces the held index sets; a reuse layer
// recomputes attention with its own q, K, V over the held sets. The sets
// stay on the device for the whole stack.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "kascade.h"

namespace kascade {

// ------------------------------------------------------------ tensor maps --
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}
}  // namespace

bool encode_tmap_2d_bf16(void* tmap, const void* base, uint64_t inner, uint64_t outer,
                         uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(reinterpret_cast<CUtensorMap*>(tmap), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Validation of a descriptor (declared in internal.h; the no-allocation
// entry point uses it too).
kascade_status check_desc(const kascade_desc* desc, Shape& s) {
  if (desc == nullptr) return KASCADE_ERR_INVALID_ARG;
  s.B = desc->batch;
  s.Hq = desc->n_q_heads;
  s.Hkv = desc->n_kv_heads;
  s.d = desc->head_dim;
  s.N = desc->kv_len;
  s.dtype = desc->dtype;
  if (s.B < 1 || s.Hkv < 1 || s.Hq < 1 || s.N < 1) return KASCADE_ERR_INVALID_ARG;
  if (s.Hq % s.Hkv != 0 || s.Hq > kMaxQHeads) return KASCADE_ERR_INVALID_ARG;
  if (s.dtype != KASCADE_F32 && s.dtype != KASCADE_BF16) return KASCADE_ERR_INVALID_ARG;
  if (s.d != 64 && s.d != 128) return KASCADE_ERR_UNSUPPORTED;
  s.G = s.Hq / s.Hkv;
  if (s.G != 1 && s.G != 2 && s.G != 4 && s.G != 8) return KASCADE_ERR_UNSUPPORTED;
  if (static_cast<long long>(s.B) * s.Hkv * s.N >= (1ll << 31)) return KASCADE_ERR_UNSUPPORTED;
  if (s.B * s.Hkv > kMaxCounterUnits) return KASCADE_ERR_UNSUPPORTED;
  if (s.N >= (1 << 24)) return KASCADE_ERR_UNSUPPORTED;
  s.scale = desc->scale > 0.f ? desc->scale : 1.0f / sqrtf(static_cast<float>(s.d));
  if (desc->index_mode != KASCADE_IDX_PER_QHEAD && desc->index_mode != KASCADE_IDX_PER_KVHEAD)
    return KASCADE_ERR_INVALID_ARG;
  s.pooled = desc->index_mode == KASCADE_IDX_PER_KVHEAD ? 1 : 0;
  s.H_idx = s.pooled ? s.Hkv : s.Hq;
  int fill[kMaxQHeads];
  for (int g = 0; g < s.Hkv; ++g) fill[g] = 0;
  for (int h = 0; h < s.Hq; ++h) {
    const int g = desc->group_map ? desc->group_map[h] : h / s.G;
    if (g < 0 || g >= s.Hkv) return KASCADE_ERR_INVALID_ARG;
    if (fill[g] >= s.G) return KASCADE_ERR_INVALID_ARG;   // unbalanced map
    s.heads[g * s.G + fill[g]++] = static_cast<int16_t>(h);
    s.head_kv[h] = static_cast<int16_t>(g);
  }
  return KASCADE_OK;
}


namespace {

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Workspace layout; offsets in bytes from the workspace base.
struct Layout {
  size_t counters, part, spill, plan, plan_count;   // decode
  size_t bracket, fcount, flist, fsamp;             // decode, fused anchor Top-k
  size_t selbits;                                   // decode: the anchor rows' selection bitmaps
  size_t row_stat, pool;                            // decode, pooled sets
  size_t lse, w, w_pool;                            // prefill (w_pool: pooled sets)
  size_t total;
};

Layout layout(const Shape& s, int topk, int mode) {
  Layout L{};
  L.counters = sizeof(WsHeader);
  size_t off = kWsStateBytes;
  if (mode == KASCADE_DECODE) {
    L.part = off;
    off = align256(off + static_cast<size_t>(s.B) * s.Hq * kMaxSplits * (s.d + 4) * 4);
    L.spill = off;
    off = align256(off + static_cast<size_t>(s.B) * s.Hq * s.N * 4);
    const size_t chunks = decode_union_chunks(s.B * s.Hkv, s.N);
    L.plan = off;
    off = align256(off + static_cast<size_t>(s.B) * s.Hkv * chunks * kPlanCapEntries * 4);
    L.plan_count = off;
    off = align256(off + static_cast<size_t>(s.B) * s.Hkv * chunks * 4);
    if (!s.pooled && s.dtype == KASCADE_BF16) {
      // fused anchor Top-k: per logit row a bracket, and per (row, split,
      // consumer warp) a sub-list of (key, position) pairs and its length
      const size_t rows = static_cast<size_t>(s.B) * s.Hq;
      const int chunk = decode_chunk_dense(s.B * s.Hkv, s.N);
      const int splits = (s.N + chunk - 1) / chunk;
      L.bracket = off;
      off = align256(off + rows * 8);
      L.fsamp = off;
      off = align256(off + rows * anchor_sample_stride(s.N) * 4);
      L.fcount = off;
      off = align256(off + rows * splits * kDecodeConsumerWarps * 4);
      L.flist = off;
      off = align256(off + rows * splits * static_cast<size_t>(chunk) * 8);
      // the anchor's selection per logit row as a bitmap, from which a layer
      // stack builds the reuse layers' union plan without searching the sets
      L.selbits = off;
      off = align256(off + rows * static_cast<size_t>((s.N + 31) / 32) * 4);
    }
    if (s.pooled) {
      L.row_stat = off;
      off = align256(off + static_cast<size_t>(s.B) * s.Hq * 8);
      L.pool = off;
      off = align256(off + static_cast<size_t>(s.B) * s.Hkv * s.N * 4);
    }
  } else {
    const size_t nT = (s.N + 127) / 128;
    const size_t per_bh = 64 * (nT - 1) * nT + s.N;
    L.lse = off;
    off = align256(off + static_cast<size_t>(s.B) * s.Hq * s.N * 4);
    L.w = off;
    off = align256(off + static_cast<size_t>(s.B) * s.Hq * per_bh * 4);
    if (s.pooled) {
      L.w_pool = off;
      off = align256(off + static_cast<size_t>(s.B) * s.Hkv * per_bh * 4);
    }
  }
  L.total = off;
  return L;
}

kascade_status check_ws(const Shape& s, int topk, int mode, void* ws, size_t ws_bytes,
                        Layout& L) {
  L = layout(s, topk, mode);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) != 0) return KASCADE_ERR_WORKSPACE;
  if (ws_bytes < L.total) return KASCADE_ERR_WORKSPACE;
  return KASCADE_OK;
}

inline kascade_status cuda_status(cudaError_t e) {
  return e == cudaSuccess ? KASCADE_OK : KASCADE_ERR_CUDA;
}

template <typename T>
inline T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

void fill_decode_args(DecodeArgs& a, const Shape& s, const void* q, const void* k, const void* v,
                      void* out, void* ws, const Layout& L, int topk) {
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.spill = at<float>(ws, L.spill);
  a.part = at<float>(ws, L.part);
  a.counters = at<unsigned int>(ws, L.counters);
  a.err = at<unsigned int>(ws, 0);
  a.plan = at<uint32_t>(ws, L.plan);
  a.plan_count = at<int32_t>(ws, L.plan_count);
  a.plan_stride = s.G * topk;
  a.pooled = s.pooled;
  a.topk = topk;
  a.B = s.B;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.N = s.N;
  a.G = s.G;
  a.scale = s.scale;
  a.scale_log2 = s.scale * 1.4426950408889634f;
  for (int i = 0; i < s.Hq; ++i) a.heads[i] = s.heads[i];
}

}  // namespace
}  // namespace kascade

// ------------------------------------------------------- decode dispatch --
namespace kascade {
namespace {

kascade_status run_dense_decode(const Shape& s, const void* q, const void* k, const void* v,
                                void* out, void* ws, const Layout& L, int topk, float* spill,
                                cudaStream_t st, float2* row_stat = nullptr) {
  DecodeArgs a;
  fill_decode_args(a, s, q, k, v, out, ws, L, topk);
  if (spill != nullptr) a.spill = spill;
  a.row_stat = row_stat;
  if (s.dtype == KASCADE_F32)
    return cuda_status(launch_decode_generic(a, s.d, s.dtype, spill ? kAnchor : kDense, st));
  a.chunk = decode_chunk_dense(s.B * s.Hkv, s.N);
  a.S = (s.N + a.chunk - 1) / a.chunk;
  return cuda_status(launch_decode_dense_bf16(a, s.d, spill != nullptr, st));
}

kascade_status run_topk_rows(const float* scores, int rows, int n, int k, int32_t* idx,
                             unsigned int* err, cudaStream_t st, uint32_t* sel_bits = nullptr) {
  TopkArgs t{};
  t.sel_bits = sel_bits;
  t.scores = scores;
  t.idx_out = idx;
  t.err = err;
  t.rows = rows;
  t.n = n;
  t.k = k;
  t.k_stride = k;
  t.prefill_tiles = 0;
  t.tile = 128;
  const cudaError_t e = launch_topk(t, st);
  return e == cudaErrorNotSupported ? KASCADE_ERR_UNSUPPORTED : cuda_status(e);
}

kascade_status run_anchor_decode(const Shape& s, const void* q, const void* k, const void* v,
                                 int topk, void* out, int32_t* idx_out, float* scores_out,
                                 void* ws, const Layout& L, cudaStream_t st, bool fused = false) {
  if (s.pooled) {
    // logits to the workspace, then the group sums of their softmax weights
    float* spill = at<float>(ws, L.spill);
    // bf16: the attention kernel's split merge also leaves each row's softmax
    // statistics, so no separate pass over the logits computes them
    const bool bf16 = s.dtype == KASCADE_BF16;
    float2* row_stat = at<float2>(ws, L.row_stat);
    kascade_status r = run_dense_decode(s, q, k, v, out, ws, L, topk, spill, st,
                                        bf16 ? row_stat : nullptr);
    if (r != KASCADE_OK) return r;
    float* pool = scores_out ? scores_out : at<float>(ws, L.pool);
    r = cuda_status(launch_pool_decode(spill, row_stat, pool, bf16, s.heads, s.B, s.Hq, s.Hkv,
                                       s.G, s.N, st));
    if (r != KASCADE_OK) return r;
    return run_topk_rows(pool, s.B * s.Hkv, s.N, topk, idx_out, at<unsigned int>(ws, 0), st);
  }
  float* spill = scores_out ? scores_out : at<float>(ws, L.spill);
  if (fused && topk < s.N) {
    // fused: a sample bracket per row, then the attention kernel files every
    // logit at or above the bracket's lower end while it spills, and the
    // selection reads those lists instead of the rows
    uint2* bracket = at<uint2>(ws, L.bracket);
    unsigned int* fcount = at<unsigned int>(ws, L.fcount);
    uint2* flist = at<uint2>(ws, L.flist);
    kascade_status r = cuda_status(launch_anchor_bracket(q, k, s.heads, s.B, s.Hq, s.Hkv, s.N,
                                                         s.d, topk, s.scale,
                                                         at<uint32_t>(ws, L.fsamp), bracket, st));
    if (r != KASCADE_OK) return r;
    DecodeArgs a;
    fill_decode_args(a, s, q, k, v, out, ws, L, topk);
    a.spill = spill;
    a.bracket = bracket;
    a.fcount = fcount;
    a.flist = flist;
    a.chunk = decode_chunk_dense(s.B * s.Hkv, s.N);
    a.S = (s.N + a.chunk - 1) / a.chunk;
    r = cuda_status(launch_decode_dense_bf16(a, s.d, true, st, true));
    if (r != KASCADE_OK) return r;
    TopkArgs t{};
    t.scores = spill;
    t.idx_out = idx_out;
    t.err = at<unsigned int>(ws, 0);
    t.rows = s.B * s.Hq;
    t.n = s.N;
    t.k = topk;
    t.k_stride = topk;
    t.tile = 128;
    t.bracket = bracket;
    t.fcount = fcount;
    t.flist = flist;
    t.fsplits = a.S;
    t.fwarps = kDecodeConsumerWarps;
    t.fchunk = a.chunk;
    t.sel_bits = at<uint32_t>(ws, L.selbits);
    const cudaError_t e = launch_topk(t, st);
    return e == cudaErrorNotSupported ? KASCADE_ERR_UNSUPPORTED : cuda_status(e);
  }
  kascade_status r = run_dense_decode(s, q, k, v, out, ws, L, topk, spill, st);
  if (r != KASCADE_OK) return r;
  return run_topk_rows(spill, s.B * s.Hq, s.N, topk, idx_out, at<unsigned int>(ws, 0), st,
                       L.selbits ? at<uint32_t>(ws, L.selbits) : nullptr);
}

// The union plan from the selection bitmaps the last anchor decode call on
// this workspace left (per-head bf16 sets; the plan of its sets).
kascade_status run_build_plan_bits(const Shape& s, int topk, void* ws, const Layout& L,
                                   cudaStream_t st) {
  if (!L.selbits) return KASCADE_ERR_UNSUPPORTED;
  DecodeArgs a;
  fill_decode_args(a, s, nullptr, nullptr, nullptr, nullptr, ws, L, topk);
  const cudaError_t e = launch_build_union_plan_bits(a, at<uint32_t>(ws, L.selbits),
                                                     (s.N + 31) / 32, at<uint32_t>(ws, L.plan),
                                                     at<int32_t>(ws, L.plan_count), st);
  return e == cudaErrorNotSupported ? KASCADE_ERR_UNSUPPORTED : cuda_status(e);
}

// Build the per-(sequence, KV head) union of the group's sets (bf16 path).
kascade_status run_build_plan(const Shape& s, const int32_t* idx, int topk, void* ws,
                              const Layout& L, cudaStream_t st) {
  DecodeArgs a;
  fill_decode_args(a, s, nullptr, nullptr, nullptr, nullptr, ws, L, topk);
  a.idx = idx;
  const cudaError_t e =
      launch_build_union_plan(a, at<uint32_t>(ws, L.plan), at<int32_t>(ws, L.plan_count), st);
  return e == cudaErrorNotSupported ? KASCADE_ERR_UNSUPPORTED : cuda_status(e);
}

kascade_status run_reuse_decode(const Shape& s, const void* q, const void* k, const void* v,
                                int topk, const int32_t* idx, void* out, void* ws,
                                const Layout& L, bool plan_ready, cudaStream_t st) {
  DecodeArgs a;
  fill_decode_args(a, s, q, k, v, out, ws, L, topk);
  a.idx = idx;
  if (s.dtype == KASCADE_F32) return cuda_status(launch_decode_generic(a, s.d, s.dtype, kSparse, st));
  if (!plan_ready && !s.pooled) {   // pooled sets are gathered directly, with no plan
    kascade_status r = run_build_plan(s, idx, topk, ws, L, st);
    if (r != KASCADE_OK) return r;
  }
  a.S = decode_union_chunks(s.B * s.Hkv, s.N);
  if (a.S > kMaxSplits) return KASCADE_ERR_UNSUPPORTED;   // N too long for 128 chunks
  return cuda_status(launch_decode_union_bf16(a, s.d, st));
}

kascade_status check_decode_ptrs(const void* q, const void* k, const void* v, const void* out) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return KASCADE_ERR_INVALID_ARG;
  return KASCADE_OK;
}

}  // namespace
}  // namespace kascade

using namespace kascade;

extern "C" {

const char* kascade_status_string(kascade_status s) {
  switch (s) {
    case KASCADE_OK: return "ok";
    case KASCADE_ERR_INVALID_ARG: return "invalid argument";
    case KASCADE_ERR_UNSUPPORTED: return "unsupported configuration";
    case KASCADE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case KASCADE_ERR_CUDA: return "CUDA error";
    case KASCADE_ERR_BAD_INPUT: return "bad input detected on the device (NaN or index out of range)";
    case KASCADE_ERR_TIMEOUT: return "bounded device wait expired";
  }
  return "unknown status";
}

size_t kascade_workspace_size(const kascade_desc* desc, int32_t topk, int32_t mode) {
  Shape s;
  if (check_desc(desc, s) != KASCADE_OK) return 0;
  if (mode != KASCADE_DECODE && mode != KASCADE_PREFILL) return 0;
  if (topk < 1) topk = 1;
  return layout(s, topk, mode).total;
}

kascade_status kascade_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr || ws_bytes < sizeof(WsHeader)) return KASCADE_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

kascade_status kascade_device_error(void* ws, void* stream) {
  if (ws == nullptr) return KASCADE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return KASCADE_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KASCADE_ERR_CUDA;
  if (word != 0) {
    const unsigned int zero[2] = {0u, 0u};
    if (cudaMemcpy(ws, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return KASCADE_ERR_CUDA;
  }
  if (word & (1u << KASCADE_ERR_TIMEOUT)) return KASCADE_ERR_TIMEOUT;
  if (word & (1u << KASCADE_ERR_BAD_INPUT)) return KASCADE_ERR_BAD_INPUT;
  return KASCADE_OK;
}

kascade_status kascade_dense_decode(const kascade_desc* desc, const void* q, const void* k,
                                    const void* v, void* out, void* ws, size_t ws_bytes,
                                    void* stream) {
  Shape s;
  kascade_status r = check_desc(desc, s);
  if (r != KASCADE_OK) return r;
  if ((r = check_decode_ptrs(q, k, v, out)) != KASCADE_OK) return r;
  Layout L;
  if ((r = check_ws(s, 1, KASCADE_DECODE, ws, ws_bytes, L)) != KASCADE_OK) return r;
  return run_dense_decode(s, q, k, v, out, ws, L, 1, nullptr, static_cast<cudaStream_t>(stream));
}

kascade_status kascade_anchor_decode(const kascade_desc* desc, const void* q, const void* k,
                                     const void* v, int32_t topk, void* out, int32_t* idx_out,
                                     float* scores_out, void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  kascade_status r = check_desc(desc, s);
  if (r != KASCADE_OK) return r;
  if ((r = check_decode_ptrs(q, k, v, out)) != KASCADE_OK) return r;
  if (topk < 1 || topk > s.N || !aligned16(idx_out)) return KASCADE_ERR_INVALID_ARG;
  if (scores_out != nullptr && !aligned16(scores_out)) return KASCADE_ERR_INVALID_ARG;
  Layout L;
  if ((r = check_ws(s, topk, KASCADE_DECODE, ws, ws_bytes, L)) != KASCADE_OK) return r;
  return run_anchor_decode(s, q, k, v, topk, out, idx_out, scores_out, ws, L,
                           static_cast<cudaStream_t>(stream));
}

kascade_status kascade_anchor_decode_fused(const kascade_desc* desc, const void* q,
                                           const void* k, const void* v, int32_t topk, void* out,
                                           int32_t* idx_out, float* scores_out, void* ws,
                                           size_t ws_bytes, void* stream) {
  Shape s;
  kascade_status r = check_desc(desc, s);
  if (r != KASCADE_OK) return r;
  if (s.pooled || s.dtype != KASCADE_BF16) return KASCADE_ERR_UNSUPPORTED;
  if ((r = check_decode_ptrs(q, k, v, out)) != KASCADE_OK) return r;
  if (topk < 1 || topk > s.N || !aligned16(idx_out)) return KASCADE_ERR_INVALID_ARG;
  if (scores_out != nullptr && !aligned16(scores_out)) return KASCADE_ERR_INVALID_ARG;
  Layout L;
  if ((r = check_ws(s, topk, KASCADE_DECODE, ws, ws_bytes, L)) != KASCADE_OK) return r;
  return run_anchor_decode(s, q, k, v, topk, out, idx_out, scores_out, ws, L,
                           static_cast<cudaStream_t>(stream), true);
}

kascade_status kascade_reuse_decode(const kascade_desc* desc, const void* q, const void* k,
                                    const void* v, int32_t topk, const int32_t* idx, void* out,
                                    void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  kascade_status r = check_desc(desc, s);
  if (r != KASCADE_OK) return r;
  if ((r = check_decode_ptrs(q, k, v, out)) != KASCADE_OK) return r;
  if (topk < 1 || topk > s.N || !aligned16(idx)) return KASCADE_ERR_INVALID_ARG;
  Layout L;
  if ((r = check_ws(s, topk, KASCADE_DECODE, ws, ws_bytes, L)) != KASCADE_OK) return r;
  return run_reuse_decode(s, q, k, v, topk, idx, out, ws, L, false,
                          static_cast<cudaStream_t>(stream));
}

kascade_status kascade_topk(const float* scores, int32_t rows, int32_t n, int32_t k,
                            int32_t* idx_out, void* ws, size_t ws_bytes, void* stream) {
  if (rows < 0 || n < 1 || k < 1 || k > n) return KASCADE_ERR_INVALID_ARG;
  if (rows > 0 && (scores == nullptr || idx_out == nullptr)) return KASCADE_ERR_INVALID_ARG;
  if (ws == nullptr || ws_bytes < sizeof(WsHeader)) return KASCADE_ERR_WORKSPACE;
  return run_topk_rows(scores, rows, n, k, idx_out, static_cast<unsigned int*>(ws),
                       static_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ------------------------------------------- sequence-sharded anchor decode --
extern "C" {

kascade_status kascade_anchor_decode_shard(const kascade_desc* desc, const void* q,
                                           const void* k, const void* v, int32_t key_offset,
                                           int32_t topk, void* out, float* lse_out,
                                           int32_t* cand_idx, float* cand_scores, void* ws,
                                           size_t ws_bytes, void* stream) {
  Shape s;
  kascade_status r = check_desc(desc, s);
  if (r != KASCADE_OK) return r;
  if (s.pooled) return KASCADE_ERR_UNSUPPORTED;
  if ((r = check_decode_ptrs(q, k, v, out)) != KASCADE_OK) return r;
  if (topk < 1 || topk > s.N || key_offset < 0 ||
      static_cast<long long>(key_offset) + s.N > 0x7fffffffll)
    return KASCADE_ERR_INVALID_ARG;
  if (!aligned16(lse_out) || !aligned16(cand_idx) || !aligned16(cand_scores))
    return KASCADE_ERR_INVALID_ARG;
  Layout L;
  if ((r = check_ws(s, topk, KASCADE_DECODE, ws, ws_bytes, L)) != KASCADE_OK) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the shard's own anchor layer: exact output, logits in the workspace spill,
  // local Top-k in cand_idx
  r = run_anchor_decode(s, q, k, v, topk, out, cand_idx, nullptr, ws, L, st);
  if (r != KASCADE_OK) return r;
  const int rows = s.B * s.Hq;
  // the split partials are free once the attention kernel is done: they hold
  // the row statistics (max, 1/sum exp) of the logits
  float2* stat = at<float2>(ws, L.part);
  const float* spill = at<float>(ws, L.spill);
  if (launch_row_stat(spill, rows, s.N, stat, st) != cudaSuccess) return KASCADE_ERR_CUDA;
  return cuda_status(launch_shard_finish(spill, stat, rows, s.N, topk, key_offset, lse_out,
                                         cand_idx, cand_scores, st));
}

size_t kascade_merge_workspace_size(const kascade_desc* desc, int32_t n_shards, int32_t topk) {
  Shape s;
  if (check_desc(desc, s) != KASCADE_OK || n_shards < 1 || topk < 1) return 0;
  const size_t rows = static_cast<size_t>(s.B) * s.Hq;
  return kWsStateBytes + align256(rows * n_shards * topk * 4) + align256(rows * topk * 4);
}

kascade_status kascade_merge_decode_shards(const kascade_desc* desc, int32_t n_shards,
                                           const void* outs, const float* lses,
                                           const int32_t* cand_idx, const float* cand_scores,
                                           int32_t topk, void* out, int32_t* idx_out, void* ws,
                                           size_t ws_bytes, void* stream) {
  Shape s;
  kascade_status r = check_desc(desc, s);
  if (r != KASCADE_OK) return r;
  if (s.pooled) return KASCADE_ERR_UNSUPPORTED;
  if (n_shards < 1 || n_shards > kMaxShards || topk < 1 || topk > s.N ||
      static_cast<long long>(n_shards) * topk >= (1ll << 24))
    return KASCADE_ERR_INVALID_ARG;
  if (!aligned16(outs) || !aligned16(lses) || !aligned16(cand_idx) || !aligned16(cand_scores) ||
      !aligned16(out) || !aligned16(idx_out))
    return KASCADE_ERR_INVALID_ARG;
  const size_t need = kascade_merge_workspace_size(desc, n_shards, topk);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) != 0 || ws_bytes < need)
    return KASCADE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int rows = s.B * s.Hq;
  const int n = n_shards * topk;
  float* scores = at<float>(ws, kWsStateBytes);
  int32_t* pos = at<int32_t>(ws, kWsStateBytes + align256(static_cast<size_t>(rows) * n * 4));
  unsigned int* err = at<unsigned int>(ws, 0);
  if ((r = cuda_status(launch_merge_out(outs, lses, n_shards, rows, s.d, s.dtype, out, st))) !=
      KASCADE_OK)
    return r;
  if ((r = cuda_status(launch_merge_scores(cand_idx, cand_scores, n_shards, rows, topk, s.N,
                                           scores, err, st))) != KASCADE_OK)
    return r;
  if ((r = run_topk_rows(scores, rows, n, topk, pos, err, st)) != KASCADE_OK) return r;
  return cuda_status(launch_merge_emit(pos, cand_idx, rows, topk, idx_out, st));
}

}  // extern "C"

// ------------------------------------------------------ prefill dispatch --
namespace kascade {
namespace {

inline kascade_status launch_status(cudaError_t e) {
  if (e == cudaErrorNotSupported) return KASCADE_ERR_UNSUPPORTED;
  return cuda_status(e);
}

void fill_prefill_args(PrefillArgs& a, const Shape& s, const void* q, const void* k,
                       const void* v, void* out, void* ws, const Layout& L, int topk) {
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = at<float>(ws, L.lse);
  a.w = at<float>(ws, L.w);
  a.err = at<unsigned int>(ws, 0);
  a.B = s.B;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.N = s.N;
  a.G = s.G;
  a.pooled = s.pooled;
  a.topk = topk;
  a.nT = (s.N + 127) / 128;
  a.scale = s.scale;
  a.scale_log2 = s.scale * 1.4426950408889634f;
  for (int h = 0; h < s.Hq; ++h) {
    a.head_kv[h] = s.head_kv[h];
    a.heads[h] = s.heads[h];
  }
}

kascade_status run_dense_prefill(const Shape& s, const void* q, const void* k, const void* v,
                                 void* out, void* ws, const Layout& L, cudaStream_t st) {
  PrefillArgs a;
  fill_prefill_args(a, s, q, k, v, out, ws, L, 1);
  return launch_status(launch_prefill_dense(a, s.d, st));
}

kascade_status run_anchor_prefill(const Shape& s, const void* q, const void* k, const void* v,
                                  int topk, void* out, int32_t* idx_out, float* weights_out,
                                  void* ws, const Layout& L, cudaStream_t st) {
  PrefillArgs a;
  fill_prefill_args(a, s, q, k, v, out, ws, L, topk);
  // per-head weights go to the caller's buffer when it asked for them (and
  // the selection reads them there); pooled sets keep the per-head weights
  // in the workspace and hand out the group sums
  if (weights_out != nullptr && !s.pooled) a.w = weights_out;
  kascade_status r = launch_status(launch_prefill_lse(a, s.d, st));
  if (r != KASCADE_OK) return r;
  if ((r = launch_status(launch_prefill_anchor_main(a, s.d, st))) != KASCADE_OK) return r;
  const float* scores = a.w;
  if (s.pooled) {
    const size_t per_bh = static_cast<size_t>(64) * (a.nT - 1) * a.nT + s.N;
    float* w_pool = weights_out != nullptr ? weights_out : at<float>(ws, L.w_pool);
    r = cuda_status(launch_pool_prefill(a.w, w_pool, s.heads, s.B, s.Hq, s.Hkv, s.G, per_bh, st));
    if (r != KASCADE_OK) return r;
    scores = w_pool;
  }
  TopkArgs t{};
  t.scores = scores;
  t.idx_out = idx_out;
  t.err = a.err;
  t.rows = s.B * s.H_idx * a.nT;
  t.n = s.N;
  t.k = topk;
  t.k_stride = topk;
  t.prefill_tiles = a.nT;
  t.tile = 128;
  return cuda_status(launch_topk(t, st));
}

kascade_status run_reuse_prefill(const Shape& s, const void* q, const void* k, const void* v,
                                 int topk, const int32_t* idx, void* out, void* ws,
                                 const Layout& L, cudaStream_t st) {
  PrefillArgs a;
  fill_prefill_args(a, s, q, k, v, out, ws, L, topk);
  a.idx = idx;
  return launch_status(launch_prefill_reuse(a, s.d, st));
}

kascade_status check_prefill(const kascade_desc* desc, Shape& s, const void* q, const void* k,
                             const void* v, const void* out) {
  kascade_status r = check_desc(desc, s);
  if (r != KASCADE_OK) return r;
  if (s.dtype != KASCADE_BF16) return KASCADE_ERR_UNSUPPORTED;
  // the prefill kernels address rows of q and out (B*Hq*N of them) with
  // 32-bit tensor-map coordinates
  if (static_cast<long long>(s.B) * s.Hq * s.N >= (1ll << 31)) return KASCADE_ERR_UNSUPPORTED;
  return check_decode_ptrs(q, k, v, out);
}

}  // namespace
}  // namespace kascade

extern "C" {

kascade_status kascade_dense_prefill(const kascade_desc* desc, const void* q, const void* k,
                                     const void* v, void* out, void* ws, size_t ws_bytes,
                                     void* stream) {
  Shape s;
  kascade_status r = check_prefill(desc, s, q, k, v, out);
  if (r != KASCADE_OK) return r;
  Layout L;
  if ((r = check_ws(s, 1, KASCADE_PREFILL, ws, ws_bytes, L)) != KASCADE_OK) return r;
  return run_dense_prefill(s, q, k, v, out, ws, L, static_cast<cudaStream_t>(stream));
}

kascade_status kascade_anchor_prefill(const kascade_desc* desc, const void* q, const void* k,
                                      const void* v, int32_t topk, void* out, int32_t* idx_out,
                                      float* weights_out, void* ws, size_t ws_bytes,
                                      void* stream) {
  Shape s;
  kascade_status r = check_prefill(desc, s, q, k, v, out);
  if (r != KASCADE_OK) return r;
  if (topk < 1 || topk > s.N || !aligned16(idx_out)) return KASCADE_ERR_INVALID_ARG;
  if (weights_out != nullptr && !aligned16(weights_out)) return KASCADE_ERR_INVALID_ARG;
  Layout L;
  if ((r = check_ws(s, topk, KASCADE_PREFILL, ws, ws_bytes, L)) != KASCADE_OK) return r;
  return run_anchor_prefill(s, q, k, v, topk, out, idx_out, weights_out, ws, L,
                            static_cast<cudaStream_t>(stream));
}

kascade_status kascade_reuse_prefill(const kascade_desc* desc, const void* q, const void* k,
                                     const void* v, int32_t topk, const int32_t* idx, void* out,
                                     void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  kascade_status r = check_prefill(desc, s, q, k, v, out);
  if (r != KASCADE_OK) return r;
  if (topk < 1 || topk > s.N || !aligned16(idx)) return KASCADE_ERR_INVALID_ARG;
  Layout L;
  if ((r = check_ws(s, topk, KASCADE_PREFILL, ws, ws_bytes, L)) != KASCADE_OK) return r;
  return run_reuse_prefill(s, q, k, v, topk, idx, out, ws, L, static_cast<cudaStream_t>(stream));
}

kascade_status kascade_run_stack_profiled(const kascade_desc* desc, int32_t mode,
                                          int32_t n_layers, const void* const* q,
                                          const void* const* k, const void* const* v,
                                          int32_t topk, const int32_t* anchors,
                                          int32_t n_anchors, void* const* out, int32_t* idx_buf,
                                          void* ws, size_t ws_bytes, void* stream,
                                          void* const* layer_events) {
  Shape s;
  kascade_status r = check_desc(desc, s);
  if (r != KASCADE_OK) return r;
  if (mode != KASCADE_DECODE && mode != KASCADE_PREFILL) return KASCADE_ERR_INVALID_ARG;
  if (mode == KASCADE_PREFILL && s.dtype != KASCADE_BF16) return KASCADE_ERR_UNSUPPORTED;
  if (n_layers < 1 || q == nullptr || k == nullptr || v == nullptr || out == nullptr)
    return KASCADE_ERR_INVALID_ARG;
  if (n_anchors < 0 || (n_anchors > 0 && anchors == nullptr)) return KASCADE_ERR_INVALID_ARG;
  for (int i = 0; i < n_anchors; ++i) {
    if (anchors[i] < 0 || anchors[i] >= n_layers) return KASCADE_ERR_INVALID_ARG;
    if (i > 0 && anchors[i] <= anchors[i - 1]) return KASCADE_ERR_INVALID_ARG;
  }
  if (n_anchors > 0 && (topk < 1 || topk > s.N || !aligned16(idx_buf)))
    return KASCADE_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)
    if ((r = check_decode_ptrs(q[l], k[l], v[l], out[l])) != KASCADE_OK) return r;
  const int tk = topk < 1 ? 1 : topk;
  Layout L;
  if ((r = check_ws(s, tk, mode, ws, ws_bytes, L)) != KASCADE_OK) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bool held = false;
  int next = 0;
  for (int l = 0; l < n_layers; ++l) {
    const bool is_anchor = next < n_anchors && anchors[next] == l;
    if (is_anchor) ++next;
    if (mode == KASCADE_DECODE) {
      if (is_anchor) {
        r = run_anchor_decode(s, q[l], k[l], v[l], tk, out[l], idx_buf, nullptr, ws, L, st);
        // the reuse layers' union plan, from the anchor's selection bitmaps
        if (r == KASCADE_OK && s.dtype == KASCADE_BF16 && !s.pooled)
          r = run_build_plan_bits(s, tk, ws, L, st);
        held = true;
      } else if (held) {
        r = run_reuse_decode(s, q[l], k[l], v[l], tk, idx_buf, out[l], ws, L, true, st);
      } else {
        r = run_dense_decode(s, q[l], k[l], v[l], out[l], ws, L, tk, nullptr, st);
      }
    } else {
      if (is_anchor) {
        r = run_anchor_prefill(s, q[l], k[l], v[l], tk, out[l], idx_buf, nullptr, ws, L, st);
        held = true;
      } else if (held) {
        r = run_reuse_prefill(s, q[l], k[l], v[l], tk, idx_buf, out[l], ws, L, st);
      } else {
        r = run_dense_prefill(s, q[l], k[l], v[l], out[l], ws, L, st);
      }
    }
    if (r != KASCADE_OK) return r;
    if (layer_events != nullptr && layer_events[l] != nullptr &&
        cudaEventRecord(static_cast<cudaEvent_t>(layer_events[l]), st) != cudaSuccess)
      return KASCADE_ERR_CUDA;
  }
  return KASCADE_OK;
}

kascade_status kascade_run_stack(const kascade_desc* desc, int32_t mode, int32_t n_layers,
                                 const void* const* q, const void* const* k,
                                 const void* const* v, int32_t topk, const int32_t* anchors,
                                 int32_t n_anchors, void* const* out, int32_t* idx_buf,
                                 void* ws, size_t ws_bytes, void* stream) {
  return kascade_run_stack_profiled(desc, mode, n_layers, q, k, v, topk, anchors, n_anchors,
                                    out, idx_buf, ws, ws_bytes, stream, nullptr);
}

}  // extern "C"

// ------------------------------------------------------------ calibration --
extern "C" {

size_t kascade_calibrate_workspace_size(const kascade_desc* desc, int32_t topk, int32_t n_layers) {
  Shape s;
  if (check_desc(desc, s) != KASCADE_OK || topk < 1 || n_layers < 1) return 0;
  const size_t dec = layout(s, topk, KASCADE_DECODE).total;
  const size_t ov = kascade_overlap_workspace_size(n_layers, s.B * s.H_idx, s.N);
  const size_t counts = static_cast<size_t>(n_layers) * n_layers * 8;
  return align256(dec > ov ? dec : ov) + align256(counts);
}

kascade_status kascade_calibrate(const kascade_desc* desc, int32_t n_layers,
                                 const void* const* q, const void* const* k,
                                 const void* const* v, int32_t topk, void* const* out,
                                 int32_t* sets_buf, double* sim_out, void* ws, size_t ws_bytes,
                                 void* stream) {
  Shape s;
  kascade_status r = check_desc(desc, s);
  if (r != KASCADE_OK) return r;
  if (n_layers < 1 || q == nullptr || k == nullptr || v == nullptr || out == nullptr ||
      sim_out == nullptr || !aligned16(sets_buf) || topk < 1 || topk > s.N)
    return KASCADE_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)   // every layer's pointers before any launch
    if ((r = check_decode_ptrs(q[l], k[l], v[l], out[l])) != KASCADE_OK) return r;
  const size_t need = kascade_calibrate_workspace_size(desc, topk, n_layers);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) != 0 || ws_bytes < need)
    return KASCADE_ERR_WORKSPACE;
  Layout L = layout(s, topk, KASCADE_DECODE);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t per_layer = static_cast<size_t>(s.B) * s.H_idx * topk;
  for (int l = 0; l < n_layers; ++l) {
    r = run_anchor_decode(s, q[l], k[l], v[l], topk, out[l], sets_buf + l * per_layer, nullptr,
                          ws, L, st);
    if (r != KASCADE_OK) return r;
  }
  const size_t dec = L.total;
  const size_t ov = kascade_overlap_workspace_size(n_layers, s.B * s.H_idx, s.N);
  long long* counts = reinterpret_cast<long long*>(static_cast<char*>(ws) +
                                                   align256(dec > ov ? dec : ov));
  char* base = static_cast<char*>(ws);
  cudaError_t e = launch_layer_overlap(sets_buf, n_layers, s.B * s.H_idx, topk, s.N, counts,
                                       reinterpret_cast<uint32_t*>(base + kWsStateBytes),
                                       reinterpret_cast<unsigned int*>(base), st);
  if (e != cudaSuccess) return KASCADE_ERR_CUDA;
  // the int64 counts land in the caller's float64 array (same element size)
  // and are turned into means in place
  const size_t nc = static_cast<size_t>(n_layers) * n_layers;
  static_assert(sizeof(long long) == sizeof(double), "in-place count conversion");
  e = cudaMemcpyAsync(sim_out, counts, nc * 8, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return KASCADE_ERR_CUDA;
  const double denom = static_cast<double>(s.B) * s.H_idx * topk;
  for (size_t i = 0; i < nc; ++i) {
    long long c;
    memcpy(&c, sim_out + i, sizeof(c));
    sim_out[i] = static_cast<double>(c) / denom;
  }
  return KASCADE_OK;
}

}  // extern "C"

// -------------------------------------------------- recall calibration --
namespace {
// Workspace of kascade_calibrate_recall: the decode layout, then the row
// statistics of the current layer, the per-row recall partials and the
// float64 similarity matrix.
struct RecallLayout {
  size_t stat, part, sim, total;
};
RecallLayout recall_layout(const Shape& s, int topk, int n_layers) {
  RecallLayout R{};
  const size_t rows = static_cast<size_t>(s.B) * s.Hq;
  size_t off = align256(layout(s, topk, KASCADE_DECODE).total);
  R.stat = off;
  off = align256(off + rows * 8);
  R.part = off;
  off = align256(off + static_cast<size_t>(n_layers) * n_layers * rows * 4);
  R.sim = off;
  off = align256(off + static_cast<size_t>(n_layers) * n_layers * 8);
  R.total = off;
  return R;
}
}  // namespace

extern "C" {

size_t kascade_calibrate_recall_workspace_size(const kascade_desc* desc, int32_t topk,
                                               int32_t n_layers) {
  Shape s;
  if (check_desc(desc, s) != KASCADE_OK || topk < 1 || n_layers < 1) return 0;
  return recall_layout(s, topk, n_layers).total;
}

kascade_status kascade_calibrate_recall(const kascade_desc* desc, int32_t n_layers,
                                        const void* const* q, const void* const* k,
                                        const void* const* v, int32_t topk, void* const* out,
                                        int32_t* sets_buf, double* sim_out, void* ws,
                                        size_t ws_bytes, void* stream) {
  Shape s;
  kascade_status r = check_desc(desc, s);
  if (r != KASCADE_OK) return r;
  if (n_layers < 1 || q == nullptr || k == nullptr || v == nullptr || out == nullptr ||
      sim_out == nullptr || !aligned16(sets_buf) || topk < 1 || topk > s.N)
    return KASCADE_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)   // every layer's pointers before any launch
    if ((r = check_decode_ptrs(q[l], k[l], v[l], out[l])) != KASCADE_OK) return r;
  const RecallLayout R = recall_layout(s, topk, n_layers);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) != 0 || ws_bytes < R.total)
    return KASCADE_ERR_WORKSPACE;
  Layout L = layout(s, topk, KASCADE_DECODE);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t per_layer = static_cast<size_t>(s.B) * s.H_idx * topk;
  const int rows = s.B * s.Hq;
  float* spill = at<float>(ws, L.spill);   // every anchor call leaves its logits here
  float2* stat = at<float2>(ws, R.stat);
  float* part = at<float>(ws, R.part);
  unsigned int* err = at<unsigned int>(ws, 0);
  for (int l = 0; l < n_layers; ++l) {
    r = run_anchor_decode(s, q[l], k[l], v[l], topk, out[l], sets_buf + l * per_layer, nullptr,
                          ws, L, st);
    if (r != KASCADE_OK) return r;
    if (launch_row_stat(spill, rows, s.N, stat, st) != cudaSuccess) return KASCADE_ERR_CUDA;
    if (launch_mass_recall(spill, stat, sets_buf, per_layer, topk, s.B, s.Hq, s.Hkv, s.N,
                           s.pooled, s.head_kv, l, n_layers, part, err, st) != cudaSuccess)
      return KASCADE_ERR_CUDA;
  }
  double* sim_dev = at<double>(ws, R.sim);
  if (launch_recall_reduce(part, n_layers, rows, sim_dev, st) != cudaSuccess)
    return KASCADE_ERR_CUDA;
  cudaError_t e = cudaMemcpyAsync(sim_out, sim_dev, static_cast<size_t>(n_layers) * n_layers * 8,
                                  cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? KASCADE_OK : KASCADE_ERR_CUDA;
}

}  // extern "C"
