// internal.h — launch interfaces between the C ABI layer (api.cu) and the
// kernel translation units. Plain structs of device pointers and sizes.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "kascade.h"

namespace kascade {

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel of the stream is still running, and must call
// pdl_wait() before touching memory that kernel writes or reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

constexpr int kMaxQHeads = 256;
constexpr int kMaxSplits = 128;
constexpr int kMaxShards = 1024;   // shards one merge call takes

// One decode attention layer (dense, anchor or reuse).
struct DecodeArgs {
  const void* q;            // [B,Hq,d]
  const void* k;            // [B,Hkv,N,d]
  const void* v;            // [B,Hkv,N,d]
  void* out;                // [B,Hq,d]
  float* spill;             // [B,Hq,N] scaled logits (anchor), or null
  float2* row_stat;         // [B*Hq] (max logit, 1 / sum exp(logit - max)) per row,
                            // written by the split merge (pooled anchor), or null
  float* part;              // [B*Hq][S][d+4]: m (log2 units), l, -, -, o[d]
  unsigned int* counters;   // [B*Hkv] split arrival counters (self-resetting)
  unsigned int* err;        // workspace error word
  const uint32_t* plan;     // union plan [B*Hkv][chunks][2048]: key | mask << 24
  const int32_t* plan_count;  // [B*Hkv][chunks]
  const int32_t* idx;       // sets [B,Hq,topk], or [B,Hkv,topk] when pooled
  int pooled;               // 1: one set per (sequence, KV head)
  int plan_stride;          // G * topk
  int topk;
  int B, Hq, Hkv, N, G;
  int S;                    // splits per (sequence, KV head)
  int plan_chunks;          // union plan: key-range chunks per (sequence, KV head)
  int chunks_per_cta;       // unused (kept zero)
  int chunk;                // keys (dense) per split
  float scale;              // sigma
  float scale_log2;         // sigma * log2(e)
  int16_t heads[kMaxQHeads];  // heads[g*G + slot] = query head of slot in group g
  // fused anchor decode (launch_decode_dense_bf16 with filter): every spilled
  // logit whose key is >= bracket[row].x joins a list. Each (row, split,
  // consumer warp) owns its own sub-list of chunk/NW entries (one warp sees at
  // most that many keys of a row), so no atomics are needed: flist
  // [B*Hq][S][chunk] (key, position), fcount [B*Hq][S][NW] entries written.
  const uint2* bracket;     // [B*Hq] (t_lo, t_hi)
  unsigned int* fcount;
  uint2* flist;
};

enum DecodeKind { kDense = 0, kAnchor = 1, kSparse = 2 };

// A validated descriptor plus the derived head tables.
struct Shape {
  int B, Hq, Hkv, d, N, G, dtype;
  int pooled;                    // one index set per KV head (GQA-pooled scores)
  int H_idx;                     // heads that own an index set: Hq, or Hkv when pooled
  float scale;
  int16_t heads[kMaxQHeads];     // heads[g*G + slot]
  int16_t head_kv[kMaxQHeads];   // KV head of each query head
};

// Checks a descriptor against the library's limits and fills the derived
// tables (api.cu): KASCADE_OK, KASCADE_ERR_INVALID_ARG or
// KASCADE_ERR_UNSUPPORTED.
kascade_status check_desc(const kascade_desc* desc, Shape& s);

// decode.cu
cudaError_t launch_decode_dense_bf16(const DecodeArgs& a, int head_dim, bool spill,
                                     cudaStream_t st, bool filter = false);
cudaError_t launch_decode_union_bf16(const DecodeArgs& a, int head_dim, cudaStream_t st);
// The same plan from the rows' selection bitmaps (TopkArgs::sel_bits of
// the group heads' rows, `words` words per row) instead of their index sets.
cudaError_t launch_build_union_plan_bits(const DecodeArgs& a, const uint32_t* sel, int words,
                                         uint32_t* plan, int32_t* plan_count, cudaStream_t st);
cudaError_t launch_build_union_plan(const DecodeArgs& a, uint32_t* plan, int32_t* plan_count,
                                    cudaStream_t st);
cudaError_t launch_decode_generic(const DecodeArgs& a, int head_dim, int dtype, DecodeKind kind,
                                  cudaStream_t st);
int decode_chunk_dense(int units, int N);        // keys per split (multiple of 64)
int decode_union_range(int units, int N);    // keys per reuse chunk
int decode_union_chunks(int units, int N);   // reuse CTAs per (sequence, KV head)
constexpr int kPlanCapEntries = 2048;        // union entries per chunk

// topk.cu
struct TopkArgs {
  const float* scores;     // row r starts at scores + row offset (see below)
  int32_t* idx_out;        // row r at idx_out + r * k_stride
  unsigned int* err;
  int rows;
  int n;                   // plain rows: row length; tile rows: sequence length
  int k;                   // requested k
  int k_stride;
  int prefill_tiles;       // 0: plain rows [rows, n]; >0: packed triangular tile rows
  int tile;                // prefill tile (128)
  // Fused anchor decode (plain rows only; null when unused): every score of
  // row r whose key is >= bracket[r].x was filed by the attention kernel as
  // (key, position) in one of the row's fsplits * fwarps sub-lists of
  // fchunk / fwarps entries (flist + r * fsplits * fchunk; lengths in fcount
  // [r][split][warp]). The selection is then made from the lists; the row
  // itself is read only when the bracket missed.
  const uint2* bracket;    // (t_lo, t_hi) keys per row
  const unsigned int* fcount;
  const uint2* flist;
  int fsplits, fwarps, fchunk;
  // Plain rows (null when unused): row r's selection as a bitmap of its n
  // positions, sel_bits + r * ceil(n / 32) (bit p % 32 of word p / 32).
  uint32_t* sel_bits;
};
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t st);

// Sample bracket of every decode logit row for the fused anchor decode:
// row r = (b, h) takes an evenly spaced sample of its keys (runs of 32),
// whose logits sigma q.k land in samp [B*Hq][anchor_sample_stride(N)] (as
// order-preserving keys), then (t_lo, t_hi) such that the k-th largest logit
// lies in [t_lo, t_hi] with high probability. bf16 q [B,Hq,d], k
// [B,Hkv,N,d]; heads[g*G + slot] as in DecodeArgs.
int anchor_sample_stride(int N);
cudaError_t launch_anchor_bracket(const void* q, const void* k, const int16_t* heads, int B,
                                  int Hq, int Hkv, int N, int d, int topk, float scale,
                                  uint32_t* samp, uint2* bracket, cudaStream_t st);
constexpr int kDecodeConsumerWarps = 4;   // consumer warps of the dense decode kernel

// prefill.cu
struct PrefillArgs {
  const void* q;        // [B,Hq,N,d]
  const void* k;        // [B,Hkv,N,d]
  const void* v;        // [B,Hkv,N,d]
  void* out;            // [B,Hq,N,d]
  float* lse;           // [B*Hq][N] log2-domain LSE of sigma*log2e*logits (anchor pass 1)
  float* w;             // packed tile weights [B*Hq][sum_t L_t]
  const int32_t* idx;   // [B,Hq,nT,topk] (reuse), or [B,Hkv,nT,topk] when pooled
  int pooled;           // 1: one set per (sequence, KV head, tile)
  unsigned int* err;
  int B, Hq, Hkv, N, G, topk, nT;
  float scale, scale_log2;
  int16_t head_kv[kMaxQHeads];   // KV head of each query head
  int16_t heads[kMaxQHeads];     // heads[g*G + slot] = query head of slot in group g
};
cudaError_t launch_prefill_dense(const PrefillArgs& a, int head_dim, cudaStream_t st);
cudaError_t launch_prefill_lse(const PrefillArgs& a, int head_dim, cudaStream_t st);
cudaError_t launch_prefill_anchor_main(const PrefillArgs& a, int head_dim, cudaStream_t st);
cudaError_t launch_prefill_reuse(const PrefillArgs& a, int head_dim, cudaStream_t st);

// pool.cu — GQA-pooled scores (one index set per KV head).
// Decode: w[b,g,j] = sum over the group's heads h of softmax_j(s[b,h,:]),
// from the anchor's logit spill s [B,Hq,N]; row_stat [B*Hq] holds each row's
// (max, 1/sum exp(s - max)): already when stats_given (the bf16 attention
// kernel's split merge writes it), else k_row_stat computes it first.
cudaError_t launch_pool_decode(const float* spill, float2* row_stat, float* w, bool stats_given,
                               const int16_t* heads, int B, int Hq, int Hkv, int G, int N,
                               cudaStream_t st);
// Row statistics alone: row_stat[r] = (max_j s_rj, 1 / sum_j exp(s_rj - max)).
cudaError_t launch_row_stat(const float* s, int rows, int n, float2* row_stat, cudaStream_t st);
// Prefill: packed tile-weight rows [B*Hq][per_bh] -> [B*Hkv][per_bh], each
// the sum of its group's rows.
cudaError_t launch_pool_prefill(const float* w, float* w_pool, const int16_t* heads, int B,
                                int Hq, int Hkv, int G, size_t per_bh, cudaStream_t st);

// recall.cu — attention-mass recall for the anchor DP: part[(l*L + i)*rows + r]
// = mass of layer l's softmax row r (logits in `spill`, statistics in
// row_stat) on the set of layer i for that row, i <= l; then the means over
// rows in float64, sim[i*L + l] (0 for i > l).
cudaError_t launch_mass_recall(const float* spill, const float2* row_stat, const int32_t* sets,
                               size_t per_layer, int topk, int B, int Hq, int Hkv, int N,
                               int pooled, const int16_t* head_kv, int layer, int n_layers,
                               float* part, unsigned int* err, cudaStream_t st);
cudaError_t launch_recall_reduce(const float* part, int n_layers, int rows, double* sim,
                                 cudaStream_t st);

// shard.cu — sequence-sharded anchor decode. A shard's partials: lse_out[r]
// from row_stat (max, 1/sum exp), and the local Top-k in cand_idx turned into
// global positions (+ offset) with their logits from the spill [rows][n_s].
cudaError_t launch_shard_finish(const float* spill, const float2* row_stat, int rows, int n_s,
                                int topk, int offset, float* lse_out, int32_t* cand_idx,
                                float* cand_scores, cudaStream_t st);
// Merge of S shards' partials (outs [S][rows][d] of dtype, lses [S][rows]).
cudaError_t launch_merge_out(const void* outs, const float* lses, int n_shards, int rows, int d,
                             int dtype, void* out, cudaStream_t st);
// scores [rows][S*topk] from cand_scores [S][rows][topk]; checks cand_idx.
cudaError_t launch_merge_scores(const int32_t* cand_idx, const float* cand_scores, int n_shards,
                                int rows, int topk, int n_total, float* scores,
                                unsigned int* err, cudaStream_t st);
// idx_out[r][i] = cand_idx of candidate pos[r][i] (a position in the row above).
cudaError_t launch_merge_emit(const int32_t* pos, const int32_t* cand_idx, int rows, int topk,
                              int32_t* idx_out, cudaStream_t st);

// overlap.cu
cudaError_t launch_layer_overlap(const int32_t* sets, int L, int units, int topk, int n_bits,
                                 long long* counts, uint32_t* bitmaps, unsigned int* err,
                                 cudaStream_t st);

// Encoding of 2-D bf16 tensor maps (api.cu owns the driver entry point).
bool encode_tmap_2d_bf16(void* tmap, const void* base, uint64_t inner, uint64_t outer,
                         uint32_t box_inner, uint32_t box_outer, bool swizzle128);

}  // namespace kascade
