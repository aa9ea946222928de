/*
 * kascade.h — C ABI of libkascade: head-aware Top-k sparse attention with
 * cross-layer index reuse (Kascade) on one GB300 GPU (sm_103a).
 *
 * Method (Kascade: A Practical Sparse Attention Method for Long-Context LLM
 * Inference; euno.news summary, sections Key Contributions and Methodology;
 * opentrain.ai page, Abstract):
 *   - anchor layers compute attention exactly and take an exact Top-k of key
 *     indices per head (Methodology 2, 5);
 *   - reuse layers recompute attention with their own q, K, V, the softmax
 *     restricted to the saved indices (Methodology 3);
 *   - prefill works per query tile (Abstract, "tile-level operations"): one
 *     index set per (head, 128-row tile), ranked by the tile's summed
 *     post-softmax weights, capped at the tile's causal prefix;
 *   - anchors are chosen offline by a DP that maximises cross-layer Top-k
 *     overlap (Key Contributions, Methodology 4).
 *
 * Conventions for every entry point
 *   - Device pointers are plain CUDA device addresses; the caller owns every
 *     buffer. The library never allocates or frees device memory.
 *   - Tensors are dense, row-major ("C-contiguous"), and their base addresses
 *     are 16-byte aligned. Element type is given by kascade_desc.dtype for q,
 *     k, v and out (bf16 or fp32); indices are int32; scores are fp32.
 *   - Layouts (B batch, Hq query heads, Hkv KV heads, N length, d head_dim):
 *       decode : q [B,Hq,d]   k,v [B,Hkv,N,d]   out [B,Hq,d]
 *                idx [B,Hq,topk]            ascending key positions
 *       prefill: q [B,Hq,N,d] k,v [B,Hkv,N,d]   out [B,Hq,N,d]
 *                idx [B,Hq,nT,topk], nT = ceil(N/128); row t holds
 *                k_t = min(topk, min(N,128(t+1))) ascending positions, then
 *                -1 padding.
 *   - Top-k rule: larger score first, lower index wins a tie, -0 == +0.
 *     Decode ranks the scaled logits sigma*q.k (the same set as ranking the
 *     softmax weights); prefill ranks the tile weights
 *     w_j = sum_{i in tile, i >= j} softmax_i(j).
 *   - `ws` is a caller-owned device workspace of at least
 *     kascade_workspace_size() bytes, 256-byte aligned. It must be zeroed
 *     once (kascade_workspace_init) before first use; afterwards the library
 *     leaves it in a reusable state: its first 65,792 bytes (error word and
 *     split counters) stay zero between calls of any shape or entry point,
 *     and must not be written by the caller. Calls sharing one workspace must
 *     be ordered (same stream, or synchronised).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream). Argument errors are returned before anything is
 *     launched; launch failures return KASCADE_ERR_CUDA. Faults found on the
 *     device (NaN scores, an out-of-range index, an expired bounded wait) are
 *     recorded in the workspace and read by kascade_device_error().
 *   - No entry point throws, blocks on the device (except
 *     kascade_device_error) or keeps pointers after it returns.
 */
#ifndef KASCADE_H
#define KASCADE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KASCADE_OK = 0,
  KASCADE_ERR_INVALID_ARG = 1,  /* bad shape, pointer, alignment, k, schedule */
  KASCADE_ERR_UNSUPPORTED = 2,  /* valid but not built: head_dim, dtype, group size */
  KASCADE_ERR_WORKSPACE = 3,    /* workspace missing or too small */
  KASCADE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  KASCADE_ERR_BAD_INPUT = 5,    /* device-detected: NaN score or index out of range */
  KASCADE_ERR_TIMEOUT = 6       /* device-detected: a bounded wait expired */
} kascade_status;

typedef enum { KASCADE_F32 = 0, KASCADE_BF16 = 1 } kascade_dtype;
typedef enum { KASCADE_DECODE = 0, KASCADE_PREFILL = 1 } kascade_mode;

/* Granularity of the index sets. The pages give every attention head its own
 * Top-k list (euno.news summary, Methodology 5); for GQA models the library
 * also offers one list per KV head ("pooled"): key j's score is the sum over
 * the group's query heads h of their softmax weights p_hj (decode) or tile
 * weights w_{t,h,j} (prefill), and every head of the group attends over the
 * group's set. Index layouts then use Hkv in place of Hq:
 *   decode idx [B,Hkv,topk], prefill idx [B,Hkv,nT,topk]. */
typedef enum { KASCADE_IDX_PER_QHEAD = 0, KASCADE_IDX_PER_KVHEAD = 1 } kascade_index_mode;

/* Shape and numerics of one attention layer. */
typedef struct {
  int32_t batch;        /* B >= 1 */
  int32_t n_q_heads;    /* Hq, a multiple of n_kv_heads, <= 256 */
  int32_t n_kv_heads;   /* Hkv >= 1 */
  int32_t head_dim;     /* d: 64 or 128 */
  int32_t kv_len;       /* N: cached keys (decode) or sequence length (prefill) */
  int32_t dtype;        /* kascade_dtype of q, k, v, out; prefill needs BF16 */
  float scale;          /* sigma; <= 0 selects 1/sqrt(head_dim) */
  /* Host array [n_q_heads]: KV head read by each query head (GQA), or NULL
   * for h / (Hq/Hkv). Every KV head must serve exactly Hq/Hkv query heads;
   * group sizes 1, 2, 4 and 8 are built. Read only during the call. */
  const int32_t* group_map;
  int32_t index_mode;   /* kascade_index_mode; 0 (zero-initialised) = per query head */
} kascade_desc;
/* Size limits (KASCADE_ERR_UNSUPPORTED beyond them): N < 2^24;
 * B*Hkv*N < 2^31; B*Hkv <= 16384; prefill also B*Hq*N < 2^31. Bf16 reuse
 * decode also needs N <= 262144 (at most 128 key-range chunks of 2048). */

/* Human-readable name of a status code (static storage). */
const char* kascade_status_string(kascade_status s);

/* Bytes of workspace the calls below need for this shape, Top-k size and
 * mode (covers every decode or prefill entry point and kascade_run_stack).
 * Returns 0 for an invalid descriptor. */
size_t kascade_workspace_size(const kascade_desc* desc, int32_t topk, int32_t mode);

/* Zero a workspace (cudaMemsetAsync on `stream`). */
kascade_status kascade_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Synchronise `stream`, then read and clear the device error word of `ws`:
 * KASCADE_OK, KASCADE_ERR_BAD_INPUT or KASCADE_ERR_TIMEOUT. */
kascade_status kascade_device_error(void* ws, void* stream);

/* Failure path of the bounded device waits, for tests: launches one wait on
 * an mbarrier that nothing completes. After the library's wait limit (about
 * two seconds) the device records KASCADE_ERR_TIMEOUT in the workspace's
 * error word (read it with kascade_device_error) and the kernel returns; the
 * context stays usable. Uses only the workspace header (>= 256 bytes). */
kascade_status kascade_check_wait_timeout(void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- decode -- */

/* Exact attention for one query per sequence over all N cached keys (the
 * library's own dense baseline; also the anchor layer's output).
 * out[b,h] = sum_j softmax_j(sigma q[b,h].k[b,g(h),j]) v[b,g(h),j]. */
kascade_status kascade_dense_decode(const kascade_desc* desc, const void* q, const void* k,
                                    const void* v, void* out, void* ws, size_t ws_bytes,
                                    void* stream);

/* Anchor layer (Methodology 2): exact output as kascade_dense_decode, and the
 * exact Top-k (1 <= topk <= N) of the scaled logits of every (sequence,
 * query head) in idx_out [B,Hq,topk], ascending. When scores_out is not NULL
 * the fp32 logits sigma*q.k are also written there, [B,Hq,N].
 * Pooled index mode: idx_out [B,Hkv,topk] is the Top-k of the pooled weights
 * w[b,g,j] = sum_{h: g(h)=g} softmax_j(sigma q[b,h].k[b,g,j]), and
 * scores_out (when not NULL) receives those fp32 weights, [B,Hkv,N]. */
kascade_status kascade_anchor_decode(const kascade_desc* desc, const void* q, const void* k,
                                     const void* v, int32_t topk, void* out, int32_t* idx_out,
                                     float* scores_out, void* ws, size_t ws_bytes, void* stream);

/* The anchor layer of kascade_anchor_decode (bf16, per query head sets; other
 * modes return KASCADE_ERR_UNSUPPORTED) with the Top-k fused into the
 * attention kernel (the logit spill fused with a threshold pass; euno.news
 * summary, Methodology 2: the anchor's exact attention and its Top-k):
 * a first kernel brackets each row's k-th logit from an evenly spaced sample
 * of its keys; the attention kernel then files every logit at or above the
 * bracket's lower end, as (key, position), in per-(row, split, warp) lists
 * while it spills, and the selection is made from those lists, re-reading a
 * row's logits only when its bracket missed (all logits equal, heavy ties, an
 * unrepresentative sample). Outputs and the index sets are identical to
 * kascade_anchor_decode's (the same fp32 logits under the same rule); on
 * GB300 the two-kernel kascade_anchor_decode is as fast or faster at the
 * measured shapes, and kascade_run_stack uses it. Same arguments and
 * workspace as kascade_anchor_decode. */
kascade_status kascade_anchor_decode_fused(const kascade_desc* desc, const void* q,
                                           const void* k, const void* v, int32_t topk, void* out,
                                           int32_t* idx_out, float* scores_out, void* ws,
                                           size_t ws_bytes, void* stream);

/* Reuse layer (Methodology 3): out[b,h] = softmax restricted to the saved set
 * S = idx[b,h,:] (topk ascending, distinct positions in [0,N)), computed with
 * this layer's q, k, v. Rows of k and v outside the sets are not read. Query
 * heads of one KV head share one pass over the union of their sets.
 * Pooled index mode: S = idx[b,g(h),:], one set per KV head. */
kascade_status kascade_reuse_decode(const kascade_desc* desc, const void* q, const void* k,
                                    const void* v, int32_t topk, const int32_t* idx, void* out,
                                    void* ws, size_t ws_bytes, void* stream);

/* Exact Top-k of fp32 rows: scores [rows, n] (row stride n) -> idx [rows,k]
 * ascending, 1 <= k <= n. A NaN anywhere sets KASCADE_ERR_BAD_INPUT on the
 * device. This is the selection the anchor calls use. Needs no workspace
 * beyond the error word (ws may be any workspace, >= 256 bytes). */
kascade_status kascade_topk(const float* scores, int32_t rows, int32_t n, int32_t k,
                            int32_t* idx_out, void* ws, size_t ws_bytes, void* stream);

/* Dense decode (as kascade_dense_decode, bf16 only) for callers that cannot
 * allocate device memory and so cannot supply a workspace: code whose device
 * memory is all owned by another allocator, or that runs where cudaMalloc is
 * not allowed. The paper has no counterpart to this entry point. Its scratch
 * (split partials, counters, error word) is a fixed 8 MiB device array inside
 * the library, held by every GPU that loads it until the process exits;
 * shapes needing more return KASCADE_ERR_WORKSPACE (the descriptor limits
 * above apply as for every entry point). The first call on a device looks
 * up the array's device address, so make it before any stream capture, and
 * do not use the library across a cudaDeviceReset. All calls share the
 * array: calls that overlap on the GPU race and must be serialised by the
 * caller. Allocates nothing. Faults found on the device (an expired bounded
 * wait) are recorded in the array's error word; kascade_noalloc_device_error
 * is the only way to read them. */
kascade_status kascade_dense_decode_noalloc(const kascade_desc* desc, const void* q,
                                            const void* k, const void* v, void* out,
                                            void* stream);

/* Synchronise `stream`, then read and clear the error word of the
 * no-allocation scratch array on the current device: KASCADE_OK,
 * KASCADE_ERR_BAD_INPUT or KASCADE_ERR_TIMEOUT. Faults of every
 * kascade_dense_decode_noalloc call since the last read accumulate there.
 * The paper has no counterpart to this entry point. Allocates nothing. */
kascade_status kascade_noalloc_device_error(void* stream);

/* ------------------------------------------ sequence-sharded anchor decode -- */
/* Context-parallel form of the anchor decode layer (Methodology 2: exact
 * attention, then an exact per-head Top-k), for a KV cache split along the
 * key axis into S contiguous shards in key order (the pages run on one
 * device and do not shard a sequence). Each shard runs
 * kascade_anchor_decode_shard on its own keys; one exchange of its partials
 * (an all-gather across the devices holding the shards) and
 * kascade_merge_decode_shards give the exact layer output and the exact
 * global Top-k: every key of the global Top-k is among its own shard's
 * Top-k, and the merge applies the same rule (larger logit first, lower
 * global position on ties) to the union. Per query head sets only
 * (index_mode 0); pooled mode returns KASCADE_ERR_UNSUPPORTED. */

/* One shard: desc->kv_len = N_s, this shard's keys; k, v [B,Hkv,N_s,d] hold
 * global positions key_offset .. key_offset + N_s - 1 (key_offset >= 0,
 * key_offset + N_s < 2^31); 1 <= topk <= N_s. Writes
 *   out         [B,Hq,d] (desc dtype): attention over the shard's keys only;
 *   lse_out     [B,Hq] fp32: log sum_j exp(s_j) over the shard, s_j = sigma q.k_j;
 *   cand_idx    [B,Hq,topk] int32: the shard's Top-k as global positions,
 *               ascending;
 *   cand_scores [B,Hq,topk] fp32: the logits s_j at those positions (the same
 *               fp32 values the unsharded anchor layer ranks).
 * ws: kascade_workspace_size(desc, topk, KASCADE_DECODE) bytes, as for
 * kascade_anchor_decode. */
kascade_status kascade_anchor_decode_shard(const kascade_desc* desc, const void* q,
                                           const void* k, const void* v, int32_t key_offset,
                                           int32_t topk, void* out, float* lse_out,
                                           int32_t* cand_idx, float* cand_scores, void* ws,
                                           size_t ws_bytes, void* stream);

/* Bytes of workspace kascade_merge_decode_shards needs (0 for an invalid
 * descriptor or sizes). */
size_t kascade_merge_workspace_size(const kascade_desc* desc, int32_t n_shards, int32_t topk);

/* Merge of n_shards (1..1024) shards' partials, shard s holding keys before
 * those of shard s + 1: desc describes the whole layer (kv_len = N, the
 * total keys; B, Hq, head_dim, dtype as the shards'). Inputs, device,
 * stacked over shards in key order: outs [S,B,Hq,d] (desc dtype), lses
 * [S,B,Hq] fp32, cand_idx [S,B,Hq,topk] int32, cand_scores [S,B,Hq,topk]
 * fp32, as kascade_anchor_decode_shard wrote them (S*topk < 2^24). Writes
 *   out     [B,Hq,d]: sum_s exp(lse_s - LSE) o_s, LSE = log sum_s exp(lse_s);
 *   idx_out [B,Hq,topk]: the global Top-k, ascending positions.
 * Candidates out of [0, N) or not ascending across the shards (shards out of
 * order), and NaN logits, set KASCADE_ERR_BAD_INPUT on the device (read with
 * kascade_device_error). */
kascade_status kascade_merge_decode_shards(const kascade_desc* desc, int32_t n_shards,
                                           const void* outs, const float* lses,
                                           const int32_t* cand_idx, const float* cand_scores,
                                           int32_t topk, void* out, int32_t* idx_out, void* ws,
                                           size_t ws_bytes, void* stream);

/* --------------------------------------------------------------- prefill -- */

/* Causal exact attention (the library's own dense baseline), bf16 only. */
kascade_status kascade_dense_prefill(const kascade_desc* desc, const void* q, const void* k,
                                     const void* v, void* out, void* ws, size_t ws_bytes,
                                     void* stream);

/* Anchor layer, prefill: exact causal output, then per (sequence, query
 * head, 128-row tile t) the Top-k_t of the tile weights w_j, k_t =
 * min(topk, L_t), L_t = min(N, 128(t+1)), into idx_out [B,Hq,nT,topk]
 * (ascending, -1 padded). Pooled index mode: per (sequence, KV head g,
 * tile) the Top-k_t of sum_{h: g(h)=g} w_{t,h,j}, idx_out [B,Hkv,nT,topk].
 * When weights_out is not NULL (16-byte aligned) the fp32 tile weights the
 * selection ranked are also written there, packed per (sequence, head):
 * [B, H, P] with P = 64*(nT-1)*nT + N (the sum of the L_t), tile t's L_t
 * weights w_0..w_{L_t-1} starting at offset 64*t*(t+1) of its (b, h) row;
 * H = Hq, or Hkv in pooled index mode (then the group sums). Feeding one
 * packed row to kascade_topk's rule reproduces idx_out exactly. */
kascade_status kascade_anchor_prefill(const kascade_desc* desc, const void* q, const void* k,
                                      const void* v, int32_t topk, void* out, int32_t* idx_out,
                                      float* weights_out, void* ws, size_t ws_bytes,
                                      void* stream);

/* Reuse layer, prefill: row i of tile t attends to S_i = {j in idx[b,h,t,:],
 * j >= 0, j <= i}; a row whose S_i is empty outputs zeros. Pooled index
 * mode: the set is idx[b,g(h),t,:]. */
kascade_status kascade_reuse_prefill(const kascade_desc* desc, const void* q, const void* k,
                                     const void* v, int32_t topk, const int32_t* idx, void* out,
                                     void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------- stack -- */

/* Run n_layers layers of one mode. q[l], k[l], v[l], out[l] are host arrays
 * of device pointers (layouts as above). anchors: host array, strictly
 * ascending layer numbers in [0, n_layers). Layer l is an anchor when listed;
 * otherwise it reuses the sets of the most recent anchor <= l, or runs dense
 * when no anchor precedes it. idx_buf (device, the decode or prefill idx
 * layout of the descriptor's index mode) holds the current sets; on return
 * it holds the last anchor's. The sets never leave the device. */
kascade_status kascade_run_stack(const kascade_desc* desc, int32_t mode, int32_t n_layers,
                                 const void* const* q, const void* const* k,
                                 const void* const* v, int32_t topk, const int32_t* anchors,
                                 int32_t n_anchors, void* const* out, int32_t* idx_buf,
                                 void* ws, size_t ws_bytes, void* stream);

/* kascade_run_stack, additionally recording layer_events[l] (a cudaEvent_t,
 * or NULL to skip) on `stream` after the launches of layer l; for per-layer
 * timing. layer_events: host array [n_layers] or NULL. */
kascade_status kascade_run_stack_profiled(const kascade_desc* desc, int32_t mode,
                                          int32_t n_layers, const void* const* q,
                                          const void* const* k, const void* const* v,
                                          int32_t topk, const int32_t* anchors,
                                          int32_t n_anchors, void* const* out, int32_t* idx_buf,
                                          void* ws, size_t ws_bytes, void* stream,
                                          void* const* layer_events);

/* ------------------------------------------------------------ scheduling -- */

/* Cross-layer Top-k overlap for the anchor DP (Methodology 4). sets: device
 * int32 [n_layers, units, topk], each row distinct positions in [0, n_bits).
 * counts_out: device int64 [n_layers, n_layers], counts_out[i][l] =
 * sum over units of |S_i ∩ S_l| (symmetric). Needs ws of
 * kascade_overlap_workspace_size bytes. */
size_t kascade_overlap_workspace_size(int32_t n_layers, int32_t units, int32_t n_bits);
kascade_status kascade_layer_overlap(const int32_t* sets, int32_t n_layers, int32_t units,
                                     int32_t topk, int32_t n_bits, int64_t* counts_out,
                                     void* ws, size_t ws_bytes, void* stream);

/* Calibration for the anchor DP (Methodology 4) on decode inputs: runs
 * every layer l as an anchor (kascade_anchor_decode) writing its exact
 * Top-k sets to sets_buf + l*B*H*topk (device int32 [n_layers, B*H,
 * topk], H = Hq, or Hkv in pooled index mode; also the layer outputs to
 * out[l]), counts the cross-layer overlaps on the device and returns
 * sim_out[i*n_layers + l] = sum over (sequence, head) of |S_i ∩ S_l| /
 * (B*H*topk) (host float64 [n_layers^2]).
 * Synchronises `stream` before returning. ws must hold
 * kascade_calibrate_workspace_size bytes. */
size_t kascade_calibrate_workspace_size(const kascade_desc* desc, int32_t topk, int32_t n_layers);
kascade_status kascade_calibrate(const kascade_desc* desc, int32_t n_layers,
                                 const void* const* q, const void* const* k,
                                 const void* const* v, int32_t topk, void* const* out,
                                 int32_t* sets_buf, double* sim_out, void* ws, size_t ws_bytes,
                                 void* stream);

/* Calibration with the attention-mass-recall similarity, an alternative to
 * the set overlap of kascade_calibrate (the pages give the DP's similarity no
 * formula; euno.news summary, Methodology 4). Every layer runs as an anchor
 * exactly as there (sets_buf and out as there) and
 *   sim_out[i*n_layers + l] = mean over (sequence, query head) of
 *                             sum_{j in S_i} softmax_j(layer l's logits),
 * for i <= l: the share of layer l's exact attention mass that the set layer
 * i holds for that head (its own set, or its KV head's in pooled index mode)
 * would keep. Entries with i > l are 0; the anchor DP reads only i <= l.
 * sim_out: host float64 [n_layers^2]. Synchronises `stream` before
 * returning. ws must hold kascade_calibrate_recall_workspace_size bytes. */
size_t kascade_calibrate_recall_workspace_size(const kascade_desc* desc, int32_t topk,
                                               int32_t n_layers);
kascade_status kascade_calibrate_recall(const kascade_desc* desc, int32_t n_layers,
                                        const void* const* q, const void* const* k,
                                        const void* const* v, int32_t topk, void* const* out,
                                        int32_t* sets_buf, double* sim_out, void* ws,
                                        size_t ws_bytes, void* stream);

/* Host DP: choose n_anchors layers (always including 0) maximising
 * F(A) = sum_l sim[a(l) * n_layers + l], a(l) = most recent anchor <= l.
 * sim: host [n_layers * n_layers], row i = anchor layer. Ties go to the
 * lexicographically smallest list. anchors_out: host [n_anchors],
 * ascending. objective_out may be NULL. */
kascade_status kascade_schedule_anchors(const double* sim, int32_t n_layers, int32_t n_anchors,
                                        int32_t* anchors_out, double* objective_out);

#ifdef __cplusplus
}
#endif
#endif /* KASCADE_H */
