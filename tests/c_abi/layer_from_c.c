/* The library used from plain C through include/moe.h only: raw device buffers, a small
 * MoE layer (route -> permute -> grouped GEMMs -> combine) with a shared expert, then
 * self-checks that need no reference implementation: the expert-major layout is a stable
 * permutation of the valid slots (cu_seqlens, src_row and inv_map agree), every token's
 * output equals the fixed-order re-sum of the layer's own rows (moe_combine_verify), and
 * the device status word stays zero.  Prints "ok" and exits 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "moe.h"

#define CHECK(x)                                                              \
  do {                                                                        \
    if (!(x)) {                                                               \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #x);        \
      return 1;                                                               \
    }                                                                         \
  } while (0)

static uint32_t lcg_state = 12345u;
static float lcg_uniform(void) { /* [-1, 1) */
  lcg_state = lcg_state * 1664525u + 1013904223u;
  return (float)(lcg_state >> 8) / 8388608.0f - 1.0f;
}
static uint16_t to_bf16(float f) { /* round to nearest even */
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
static void* upload(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes) != cudaSuccess) return NULL;
  if (cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}
static uint16_t* random_bf16(size_t n, float scale) {
  uint16_t* h = (uint16_t*)malloc(n * 2);
  for (size_t i = 0; i < n; ++i) h[i] = to_bf16(lcg_uniform() * scale);
  return h;
}

int main(void) {
  const int T = 96, H = 256, I = 128, E = 16, K = 4;
  CHECK(moe_abi_version() == 6);

  float* h_logits = (float*)malloc((size_t)T * E * 4);
  for (int i = 0; i < T * E; ++i) h_logits[i] = lcg_uniform() * 3.0f;
  uint16_t* h_x = random_bf16((size_t)T * H, 1.0f);
  uint16_t* h_w13 = random_bf16((size_t)E * 2 * I * H, 0.06f);
  uint16_t* h_w2 = random_bf16((size_t)E * H * I, 0.08f);
  uint16_t* h_s13 = random_bf16((size_t)2 * I * H, 0.06f);
  uint16_t* h_s2 = random_bf16((size_t)H * I, 0.08f);

  float* logits = (float*)upload(h_logits, (size_t)T * E * 4);
  uint16_t* x = (uint16_t*)upload(h_x, (size_t)T * H * 2);
  void* w13 = upload(h_w13, (size_t)E * 2 * I * H * 2);
  void* w2 = upload(h_w2, (size_t)E * H * I * 2);
  void* s13 = upload(h_s13, (size_t)2 * I * H * 2);
  void* s2 = upload(h_s2, (size_t)H * I * 2);
  CHECK(logits && x && w13 && w2 && s13 && s2);

  moe_layer_desc_t d;
  memset(&d, 0, sizeof d);
  d.T = T; d.H = H; d.I = I; d.E = E; d.K = K; d.dtype = MOE_BF16; d.has_shared = 1;
  moe_layer_weights_t w;
  memset(&w, 0, sizeof w);
  w.w13 = w13; w.w2 = w2; w.shared_w13 = s13; w.shared_w2 = s2;
  const size_t ws_bytes = moe_layer_workspace_bytes(&d);
  CHECK(ws_bytes > 0);
  void* ws = NULL;
  int32_t *topk_idx = NULL, *status = NULL;
  float* topk_w = NULL;
  uint16_t* out = NULL;
  CHECK(cudaMalloc(&ws, ws_bytes) == cudaSuccess);
  CHECK(cudaMalloc((void**)&topk_idx, (size_t)T * K * 4) == cudaSuccess);
  CHECK(cudaMalloc((void**)&topk_w, (size_t)T * K * 4) == cudaSuccess);
  CHECK(cudaMalloc((void**)&out, (size_t)T * H * 2) == cudaSuccess);
  CHECK(cudaMalloc((void**)&status, 4) == cudaSuccess);
  CHECK(cudaMemset(status, 0, 4) == cudaSuccess);

  CHECK(moe_layer_forward(&d, &w, logits, NULL, topk_idx, topk_w, x, NULL, NULL, out, ws, ws_bytes, status,
                          NULL) == MOE_OK);
  /* a short workspace is refused before anything is launched */
  CHECK(moe_layer_forward(&d, &w, logits, NULL, topk_idx, topk_w, x, NULL, NULL, out, ws, ws_bytes - 256,
                          status, NULL) == MOE_ERR_WORKSPACE);

  moe_layer_views_t v;
  CHECK(moe_layer_views(&d, ws, &v) == MOE_OK);
  CHECK(v.cap == T * K + T);
  /* the output is the fixed-order re-sum of the layer's own rows, for every token */
  CHECK(moe_combine_verify(v.y, v.inv_map, topk_w, T, K, H, v.y, v.shared_map, NULL, out, status, NULL) == MOE_OK);
  CHECK(cudaDeviceSynchronize() == cudaSuccess);

  int32_t h_status = -1;
  CHECK(cudaMemcpy(&h_status, status, 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(h_status == 0);

  /* the layout: cu_seqlens counts every slot (no padding here) plus one shared row per
   * token; src_row and inv_map are inverse permutations; rows of a segment hold that
   * expert's slots in ascending flat order */
  int32_t* h_idx = (int32_t*)malloc((size_t)T * K * 4);
  int32_t* h_cu = (int32_t*)malloc((size_t)(E + 2) * 4);
  int32_t* h_src = (int32_t*)malloc((size_t)v.cap * 4);
  int32_t* h_inv = (int32_t*)malloc((size_t)T * K * 4);
  CHECK(cudaMemcpy(h_idx, topk_idx, (size_t)T * K * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(cudaMemcpy(h_cu, v.cu_seqlens, (size_t)(E + 2) * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(cudaMemcpy(h_src, v.src_row, (size_t)v.cap * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(cudaMemcpy(h_inv, v.inv_map, (size_t)T * K * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(h_cu[0] == 0 && h_cu[E] == T * K && h_cu[E + 1] == T * K + T);
  for (int e = 0; e < E; ++e) {
    CHECK(h_cu[e] <= h_cu[e + 1]);
    for (int p = h_cu[e]; p < h_cu[e + 1]; ++p) {
      const int s = h_src[p];
      CHECK(s >= 0 && s < T * K && h_idx[s] == e && h_inv[s] == p);
      if (p > h_cu[e]) CHECK(h_src[p - 1] < s);
    }
  }
  for (int p = h_cu[E]; p < h_cu[E + 1]; ++p) CHECK(h_src[p] == T * K + (p - h_cu[E]));
  for (int t = 0; t < T; ++t)   /* top-k ids of a token are distinct */
    for (int a = 0; a < K; ++a)
      for (int b2 = a + 1; b2 < K; ++b2) CHECK(h_idx[t * K + a] != h_idx[t * K + b2]);

  /* the same layer on weights packed into the tile layout: the same output, bit for bit */
  void *t13 = NULL, *t2 = NULL, *ts13 = NULL, *ts2 = NULL;
  uint16_t* out_t = NULL;
  CHECK(cudaMalloc(&t13, (size_t)E * 2 * I * H * 2) == cudaSuccess);
  CHECK(cudaMalloc(&t2, (size_t)E * H * I * 2) == cudaSuccess);
  CHECK(cudaMalloc(&ts13, (size_t)2 * I * H * 2) == cudaSuccess);
  CHECK(cudaMalloc(&ts2, (size_t)H * I * 2) == cudaSuccess);
  CHECK(cudaMalloc((void**)&out_t, (size_t)T * H * 2) == cudaSuccess);
  CHECK(moe_pack_weights(w13, E, 2 * I, H, MOE_BF16, t13, NULL) == MOE_OK);
  CHECK(moe_pack_weights(w2, E, H, I, MOE_BF16, t2, NULL) == MOE_OK);
  CHECK(moe_pack_weights(s13, 1, 2 * I, H, MOE_BF16, ts13, NULL) == MOE_OK);
  CHECK(moe_pack_weights(s2, 1, H, I, MOE_BF16, ts2, NULL) == MOE_OK);
  CHECK(moe_pack_weights(w13, E, 2 * I, H, MOE_BF16, w13, NULL) == MOE_ERR_ARG);   /* not in place */
  moe_layer_desc_t dt = d;
  dt.weight_tiles = 1;
  moe_layer_weights_t wt = w;
  wt.w13 = t13; wt.w2 = t2; wt.shared_w13 = ts13; wt.shared_w2 = ts2;
  CHECK(moe_layer_forward(&dt, &wt, logits, NULL, topk_idx, topk_w, x, NULL, NULL, out_t, ws, ws_bytes, status,
                          NULL) == MOE_OK);
  uint16_t* h_out = (uint16_t*)malloc((size_t)T * H * 2);
  uint16_t* h_out_t = (uint16_t*)malloc((size_t)T * H * 2);
  CHECK(cudaMemcpy(h_out, out, (size_t)T * H * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(cudaMemcpy(h_out_t, out_t, (size_t)T * H * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(memcmp(h_out, h_out_t, (size_t)T * H * 2) == 0);
  CHECK(cudaMemcpy(&h_status, status, 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(h_status == 0);

  printf("ok\n");
  return 0;
}
