/* Plain C99 client of libkascade: includes the public header, links the
 * shared library and exercises the calls that need no GPU (argument
 * validation, workspace sizing, status strings and the host anchor DP).
 * Prints one line per check and exits non-zero on the first failure. Built
 * and run by tests/test_c_abi_host.py. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "kascade.h"

static int failures = 0;

static void expect(int ok, const char* what) {
  printf("%s %s\n", ok ? "ok" : "FAIL", what);
  if (!ok) ++failures;
}

int main(void) {
  /* a zero-initialised descriptor means per-query-head sets and 1/sqrt(d) */
  kascade_desc d;
  memset(&d, 0, sizeof(d));
  d.batch = 2;
  d.n_q_heads = 8;
  d.n_kv_heads = 2;
  d.head_dim = 128;
  d.kv_len = 4096;
  d.dtype = KASCADE_BF16;

  const size_t ws_dec = kascade_workspace_size(&d, 512, KASCADE_DECODE);
  const size_t ws_pre = kascade_workspace_size(&d, 512, KASCADE_PREFILL);
  expect(ws_dec > 0 && ws_pre > 0, "workspace sizes for a valid descriptor");
  /* the decode workspace holds at least the fp32 logit spill [B,Hq,N] */
  expect(ws_dec >= (size_t)2 * 8 * 4096 * 4, "decode workspace holds the logit spill");

  kascade_desc bad = d;
  bad.n_q_heads = 6; /* 6 query heads over 2 KV heads: group size 3 is not built */
  expect(kascade_workspace_size(&bad, 512, KASCADE_DECODE) == 0, "group size 3 refused");
  bad = d;
  bad.index_mode = 7;
  expect(kascade_workspace_size(&bad, 512, KASCADE_DECODE) == 0, "unknown index mode refused");

  /* validation happens before any launch: fake, aligned addresses are never read */
  void* p = (void*)(uintptr_t)(1u << 20);
  void* mis = (void*)(uintptr_t)((1u << 20) + 4);
  int32_t* ip = (int32_t*)p;
  expect(kascade_anchor_decode(&d, p, p, p, 0, p, ip, NULL, p, ws_dec, NULL) ==
             KASCADE_ERR_INVALID_ARG, "topk 0 refused");
  expect(kascade_anchor_decode(&d, p, p, p, 4097, p, ip, NULL, p, ws_dec, NULL) ==
             KASCADE_ERR_INVALID_ARG, "topk > N refused");
  expect(kascade_reuse_decode(&d, mis, p, p, 64, ip, p, p, ws_dec, NULL) ==
             KASCADE_ERR_INVALID_ARG, "misaligned q refused");
  expect(kascade_dense_decode(&d, p, p, p, p, p, 64, NULL) == KASCADE_ERR_WORKSPACE,
         "small workspace refused");
  expect(kascade_dense_prefill(&d, p, p, p, p, NULL, ws_pre, NULL) == KASCADE_ERR_WORKSPACE,
         "null workspace refused");
  expect(kascade_topk(p, 4, 10, 11, ip, p, 256, NULL) == KASCADE_ERR_INVALID_ARG,
         "k > n refused");
  expect(kascade_schedule_anchors(NULL, 4, 2, ip, NULL) == KASCADE_ERR_INVALID_ARG,
         "null similarity refused");
  expect(kascade_anchor_prefill(&d, p, p, p, 512, p, ip, (float*)mis, p, ws_pre, NULL) ==
             KASCADE_ERR_INVALID_ARG, "misaligned tile-weights buffer refused");
  expect(kascade_anchor_decode_shard(&d, p, p, p, -1, 512, p, (float*)p, ip, (float*)p, p,
                                     ws_dec, NULL) == KASCADE_ERR_INVALID_ARG,
         "negative shard offset refused");
  const size_t ws_merge = kascade_merge_workspace_size(&d, 4, 512);
  expect(ws_merge > 0, "merge workspace size");
  expect(kascade_merge_decode_shards(&d, 0, p, (float*)p, ip, (float*)p, 512, p, ip, p, ws_merge,
                                     NULL) == KASCADE_ERR_INVALID_ARG, "zero shards refused");
  expect(kascade_merge_decode_shards(&d, 4, p, (float*)p, ip, (float*)p, 512, p, ip, p, 256,
                                     NULL) == KASCADE_ERR_WORKSPACE, "small merge workspace refused");
  kascade_desc f32 = d;
  f32.dtype = KASCADE_F32;
  expect(kascade_anchor_decode_fused(&f32, p, p, p, 512, p, ip, NULL, p, ws_dec, NULL) ==
             KASCADE_ERR_UNSUPPORTED, "fused anchor decode needs bf16");

  for (int s = KASCADE_OK; s <= KASCADE_ERR_TIMEOUT; ++s) {
    const char* msg = kascade_status_string((kascade_status)s);
    expect(msg != NULL && msg[0] != '\0', "status string");
  }

  /* host DP on a block matrix: layers 0-3 and 4-7 agree among themselves */
  double sim[64];
  for (int i = 0; i < 8; ++i)
    for (int l = 0; l < 8; ++l) sim[i * 8 + l] = (i == l) ? 1.0 : ((i < 4) == (l < 4) ? 0.9 : 0.1);
  int32_t anchors[2] = {-1, -1};
  double obj = 0.0;
  expect(kascade_schedule_anchors(sim, 8, 2, anchors, &obj) == KASCADE_OK, "DP runs");
  expect(anchors[0] == 0 && anchors[1] == 4, "DP picks the block starts 0 and 4");
  /* F = 2 diagonal terms + 6 in-block terms of 0.9 */
  expect(fabs(obj - (2.0 + 6 * 0.9)) < 1e-12, "DP objective");
  int32_t three[3];
  expect(kascade_schedule_anchors(sim, 2, 3, three, NULL) == KASCADE_ERR_INVALID_ARG,
         "more anchors than layers refused");

  printf("%d failure(s)\n", failures);
  return failures == 0 ? 0 : 1;
}
