// Router: softmax -> top-k -> renormalise, one warp per token.
//
// The DeepEP page passes per-token topk_weights / topk_ids into dispatch and the MoonEP
// page works with [T, K] expert ids; neither defines the router function, so this takes
// the plain softmax -> top-k -> renormalise reading.  Selection happens on the float32 logits
// (softmax is monotone): descending, ties to the lower expert id, so the ids are exact.
// The renormalised weights need only the chosen logits: the full softmax denominator
// cancels, w_k = e^{l_k - l_max} / sum_j e^{l_j - l_max}.
//
// Bound: HBM, T*E*4 bytes read + T*K*8 written; one warp reads its token's E logits
// with coalesced loads (lane l holds experts l, l+32, ...).  Each of the K selection rounds
// is one 64-bit max per lane and a 5-step warp butterfly on packed (logit, id) keys.
#include "common.cuh"

namespace moe {

// Order-preserving key of (logit, expert id): the float's bits mapped so that unsigned order
// is float order in the high word, the complemented id in the low word -- so the largest
// key is the largest logit, ties going to the lower id.  0 marks an empty entry (every
// finite logit maps above it).  -0 is keyed as +0: equal floats tie on the id.
__device__ __forceinline__ unsigned long long route_key(float v, int e) {
  const uint32_t b = v == 0.0f ? 0u : __float_as_uint(v);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)ord << 32) | (uint32_t)(~e);
}
__device__ __forceinline__ float key_logit(unsigned long long k) {
  const uint32_t ord = (uint32_t)(k >> 32);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7fffffffu) : ~ord);
}

template <int EPL>  // experts per lane = ceil(E / 32)
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                         int K, const int32_t* __restrict__ num_tokens,
                                                         int32_t* __restrict__ topk_idx,
                                                         float* __restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const int n = num_tokens ? *num_tokens : T;
  if (t >= n) {
    if (lane < K) {
      topk_idx[(size_t)t * K + lane] = -1;
      topk_w[(size_t)t * K + lane] = 0.0f;
    }
    return;
  }
  unsigned long long key[EPL];
  const float* row = logits + (size_t)t * E;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = lane + 32 * j;
    key[j] = e < E ? route_key(row[e], e) : 0ull;
  }
  int my_id = -1;      // lane k keeps the k-th chosen id and logit
  float my_logit = 0.0f;
  float top_logit = 0.0f;
  for (int k = 0; k < K; ++k) {
    unsigned long long m = key[0];
#pragma unroll
    for (int j = 1; j < EPL; ++j) m = key[j] > m ? key[j] : m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, m, off);
      m = o > m ? o : m;
    }
    // m is warp-uniform: its owner clears it
#pragma unroll
    for (int j = 0; j < EPL; ++j)
      if (key[j] == m) key[j] = 0ull;
    const float lv = key_logit(m);
    if (lane == k) {
      my_id = (int)(~(uint32_t)m);
      my_logit = lv;
    }
    if (k == 0) top_logit = lv;
  }
  const float ex = (lane < K) ? expf(my_logit - top_logit) : 0.0f;
  // sum in ascending slot order (a fixed order, independent of the warp reduction tree)
  float sum = 0.0f;
  for (int k = 0; k < K; ++k) sum += __shfl_sync(0xffffffffu, ex, k);
  if (lane < K) {
    topk_idx[(size_t)t * K + lane] = my_id;
    topk_w[(size_t)t * K + lane] = __fdiv_rn(ex, sum);
  }
}

}  // namespace moe

extern "C" moe_status_t moe_route_topk(const float* logits, int T, int E, int K, const int32_t* num_tokens,
                                       int32_t* topk_idx, float* topk_w, void* stream) {
  using namespace moe;
  if (T < 0 || E < 1 || E > kMaxExperts || K < 1 || K > E || K > kMaxTopK) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_idx || !topk_w) return MOE_ERR_ARG;
  const int threads = 256;
  const int blocks = (T + 7) / 8;
  cudaStream_t s = as_stream(stream);
  const int epl = (E + 31) / 32;
  if (epl <= 1)
    route_topk_kernel<1><<<blocks, threads, 0, s>>>(logits, T, E, K, num_tokens, topk_idx, topk_w);
  else if (epl <= 2)
    route_topk_kernel<2><<<blocks, threads, 0, s>>>(logits, T, E, K, num_tokens, topk_idx, topk_w);
  else if (epl <= 4)
    route_topk_kernel<4><<<blocks, threads, 0, s>>>(logits, T, E, K, num_tokens, topk_idx, topk_w);
  else if (epl <= 8)
    route_topk_kernel<8><<<blocks, threads, 0, s>>>(logits, T, E, K, num_tokens, topk_idx, topk_w);
  else if (epl <= 16)
    route_topk_kernel<16><<<blocks, threads, 0, s>>>(logits, T, E, K, num_tokens, topk_idx, topk_w);
  else
    route_topk_kernel<32><<<blocks, threads, 0, s>>>(logits, T, E, K, num_tokens, topk_idx, topk_w);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}
