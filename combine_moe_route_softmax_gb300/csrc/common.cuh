// Shared device/host helpers of libmoe (sm_103a).  Internal header.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include <atomic>

#include "../../include/moe.h"

#define MOE_CHECK_LAUNCH()                                   \
  do {                                                       \
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

namespace moe {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;

// SM count of the current device (cached per device; 1 -- always a valid grid size -- if
// the query fails).
inline int num_sms() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  std::atomic<int>& c = cache[dev & 63];
  int n = c.load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
  c.store(n, std::memory_order_relaxed);
  return n;
}

// Function attributes live in each device's context: run `set` (returning true on success)
// once per device.  Concurrent first calls may both run it, which is harmless.
template <class F>
inline bool once_per_device(std::atomic<unsigned long long>& done, F&& set) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return true;
  if (!set()) return false;
  done.fetch_or(bit, std::memory_order_release);
  return true;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
// E4M3 (e4m3fn) round-to-nearest-even with saturation to +-448 (hardware cvt).
__device__ __forceinline__ uint8_t f32_to_e4m3(float f) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(f, __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float e4m3_to_f32(uint8_t q) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(q), __NV_E4M3);
  return __half2float(__half(h));
}
// 1xN block scale rule: s = amax / 448 (IEEE float32 division), 1 if not positive.
__device__ __forceinline__ float block_scale(float amax) {
  float s = __fdiv_rn(amax, 448.0f);
  return s > 0.0f ? s : 1.0f;
}

// E2M1 rounding of two float32 values with the hardware conversions:
// cvt.rn.satfinite.e2m1x2.f32 rounds to nearest, ties to the even code, and saturates at 6
// (0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4, 7 -> 6), packing
// its first operand in the high nibble; cvt.rn.f16x2.e2m1x2 decodes the pair exactly, high
// nibble to the high half.  Held bit for bit (and sign for sign) to an E2M1 written from
// the format's definition by the GPU tests.
__device__ __forceinline__ void e2m1_round2(float lo, float hi, float& lo_q, float& hi_q) {
  uint32_t h2;
  asm("{\n\t.reg .b8 q;\n\tcvt.rn.satfinite.e2m1x2.f32 q, %1, %2;\n\tcvt.rn.f16x2.e2m1x2 %0, q;\n\t}"
      : "=r"(h2)
      : "f"(hi), "f"(lo));
  lo_q = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
  hi_q = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// The permute behind moe_permute / moe_permute_ex / moe_permute_batched (permute.cu);
// zero_buf (nullable, [T, zero_per_token] int32) is cleared by its first kernel, for the
// layer's fused combine counters.
moe_status_t permute_impl(const int32_t* topk_idx, int T, int K, int E, int with_shared, const uint16_t* x, int H,
                          moe_dtype_t out_dtype, void* xp, float* xp_scales, int32_t* cu_seqlens, int32_t* src_row,
                          int32_t* inv_map, int32_t* shared_map, void* ws, size_t ws_bytes, int32_t* dev_status,
                          const float* dq_scale, const float* topk_w, float* row_w, int max_tokens,
                          int32_t* masked_m, void* stream, int32_t* zero_buf, int zero_per_token,
                          int dq_format = 0);

}  // namespace moe
