// FP8 E4M3 weight quantisation with one float32 scale per 128x128 block (the DeepEP
// page's block_n x block_k weight tiles): s = amax/448 (1 if not positive),
// q = e4m3_rn_satfinite(w / s).  A one-time weight-preparation call, outside the layer.
// One 256-thread block per 128x128 tile: each thread reads 64 elements as 8 16-byte
// vectors, the block reduces the tile's amax, then every thread writes its codes.
#include <algorithm>

#include "common.cuh"

namespace moe {

__global__ void __launch_bounds__(256) quant_weight_kernel(const uint16_t* __restrict__ w, int rows, int cols,
                                                           uint8_t* __restrict__ q, float* __restrict__ scales) {
  __shared__ float red[8];
  const int rb = rows / 128, cb = cols / 128;
  const int tile = blockIdx.x;
  const int m = tile / (rb * cb);
  const int r0 = ((tile / cb) % rb) * 128;
  const int c0 = (tile % cb) * 128;
  const size_t base = (size_t)m * rows * cols;
  // thread -> row (tid / 2), 64-column half (tid % 2)
  const int r = r0 + (threadIdx.x >> 1);
  const int c = c0 + (threadIdx.x & 1) * 64;
  const uint4* src = reinterpret_cast<const uint4*>(w + base + (size_t)r * cols + c);
  float f[64];
  float amax = 0.0f;
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const uint4 u = __ldg(src + v);
    const uint32_t x[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[8 * v + 2 * i] = __uint_as_float(x[i] << 16);
      f[8 * v + 2 * i + 1] = __uint_as_float(x[i] & 0xffff0000u);
    }
  }
#pragma unroll
  for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float s = block_scale(amax);
  uint4* dst = reinterpret_cast<uint4*>(q + base + (size_t)r * cols + c);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t word = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) word |= (uint32_t)f32_to_e4m3(__fdiv_rn(f[16 * v + 4 * j + b], s)) << (8 * b);
      o[j] = word;
    }
    dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (threadIdx.x == 0) scales[(size_t)m * rb * cb + (size_t)(r0 / 128) * cb + c0 / 128] = s;
}

}  // namespace moe

namespace moe {
// max |x| over a BF16 tensor -> atomicMax on the float bits of *amax (non-negative floats
// order like their bit patterns as signed ints).
__global__ void __launch_bounds__(256) amax_bf16_kernel(const uint16_t* __restrict__ x, size_t n,
                                                        float* __restrict__ amax) {
  float m = 0.0f;
  const size_t nv = n / 8;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x; v < nv; v += stride) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(x) + v);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xffff0000u))));
  }
  for (size_t i = nv * 8 + (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    m = fmaxf(m, fabsf(bf16_to_f32(x[i])));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0 && m > 0.0f) atomicMax(reinterpret_cast<int*>(amax), __float_as_int(m));
}
}  // namespace moe

extern "C" moe_status_t moe_amax_bf16(const uint16_t* x, size_t n, float* amax, void* stream) {
  using namespace moe;
  if (!amax || (n > 0 && !x) || (reinterpret_cast<uintptr_t>(x) & 15)) return MOE_ERR_ARG;
  if (n == 0) return MOE_OK;
  const size_t blocks = std::min<size_t>((n / 8 + 255) / 256 + 1, (size_t)num_sms() * 8);
  amax_bf16_kernel<<<(unsigned)blocks, 256, 0, as_stream(stream)>>>(x, n, amax);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

extern "C" moe_status_t moe_quantize_weight_fp8(const uint16_t* w, int mats, int rows, int cols, uint8_t* q,
                                                float* scales, void* stream) {
  using namespace moe;
  if (mats < 0 || rows <= 0 || cols <= 0 || rows % 128 != 0 || cols % 128 != 0) return MOE_ERR_ARG;
  if (mats == 0) return MOE_OK;
  if (!w || !q || !scales) return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(q)) & 15) return MOE_ERR_ARG;
  const size_t tiles = (size_t)mats * (rows / 128) * (cols / 128);
  if (tiles > 0x7fffffffull) return MOE_ERR_ARG;
  quant_weight_kernel<<<(unsigned)tiles, 256, 0, as_stream(stream)>>>(w, rows, cols, q, scales);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

extern "C" int moe_abi_version(void) { return 6; }

extern "C" const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}
