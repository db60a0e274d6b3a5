// Combine: gather each token's K expert rows through the inverse map, router-weight
// them, optionally fake-quantise each weighted row to E4M3 with a constant scale, sum in
// float32 in ascending slot order starting from +0, add the shared expert's row last and
// unquantised, round once to BF16.
//
// Mega-MoE page: the combine fake-quantiser acts on the router-weighted per-(token,
// slot) rows and then re-adds them exactly as the fused kernel does -- slots in increasing
// order, a float32 accumulator starting at zero, a single rounding to BF16, the fused
// shared expert last and never quantised.  The same page checks once that such a re-sum
// equals the kernel's output exactly, and inside a captured graph does the comparison on
// the device (here moe_combine_verify, which reports through a status word instead of an
// assert).
//
// Every float op is an explicit round-to-nearest intrinsic (__fmul_rn / __fadd_rn /
// __fdiv_rn) so the compiler cannot contract them into FMAs: the result is bit-exact
// against a float32 reference fed the same rows.  The fake-quant's division by s runs once
// per E4M3 code into a shared-memory table, not once per element.
//
// One warp per (token, column part); lane l owns 16-byte vectors l, l+32, ... of the
// part.  A token's row is split into `splits` parts only when there are too few tokens
// to fill the GPU (decode: 128 tokens); the order of the sum is per element, so the split
// changes nothing in the result.  For each vector, the K slot rows are loaded together
// (up to 8 16-byte loads in flight per lane) before the ordered sum.  HBM-bound:
// N*H*2 + N_shared*H*2 read, T*H*2 written.
#include "common.cuh"

namespace moe {

enum CombineMode { kWrite = 0, kVerify = 1, kAmax = 2 };

// K <= 8: at most 64 registers, so 4 blocks (32 warps) per SM keep enough loads in flight.
// SPLIT = false (enough tokens) is the plain warp-per-token loop.
template <int MODE, bool FQ, int KMAX, bool SPLIT>
__global__ void __launch_bounds__(256) combine_kernel(
    const uint16_t* __restrict__ y, const int32_t* __restrict__ inv_map, const float* __restrict__ topk_w, int T,
    int K, int H, const uint16_t* __restrict__ shared_y, const int32_t* __restrict__ shared_map,
    const float* __restrict__ fq_scale, uint16_t* __restrict__ out, const uint16_t* __restrict__ expected,
    int32_t* dev_status, float* amax_out, int splits) {
  const int lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int nvec = H / 8;
  const int per_part = SPLIT ? (nvec + splits - 1) / splits : nvec;
  const float s = FQ ? *fq_scale : 1.0f;
  // fake-quant dequantisation table: code -> fl32(decode(code) / s), the same IEEE divisions
  // the per-element QDQ would do (s is one scalar), made once per block
  __shared__ float fq_tbl[FQ ? 256 : 1];
  if (FQ) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) fq_tbl[i] = __fdiv_rn(e4m3_to_f32((uint8_t)i), s);
    __syncthreads();
  }
  float amax = 0.0f;
  bool mismatch = false;
  const int n_items = SPLIT ? T * splits : T;
  for (int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < n_items; item += nw) {
    const int t = SPLIT ? item / splits : item;
    const int v_begin = SPLIT ? (item - t * splits) * per_part : 0;
    const int v_end = SPLIT ? min(nvec, v_begin + per_part) : nvec;
    int my_p = -1;
    float my_w = 0.0f;
    if (lane < K) {
      my_p = inv_map[(size_t)t * K + lane];
      my_w = topk_w ? topk_w[(size_t)t * K + lane] : 1.0f;   // NULL: rows already weighted
    }
    const unsigned valid = __ballot_sync(0xffffffffu, lane < K && my_p >= 0);
    int srow = -1;
    if (MODE != kAmax && valid && shared_y) srow = shared_map ? shared_map[t] : t;
    int p[KMAX];
    float w[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      p[j] = __shfl_sync(0xffffffffu, my_p, j);
      w[j] = __shfl_sync(0xffffffffu, my_w, j);
      if (j >= K) p[j] = -1;
    }
    for (int v = v_begin + lane; v < v_end; v += 32) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      uint4 ld[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (p[j] >= 0) ld[j] = __ldg(reinterpret_cast<const uint4*>(y + (size_t)p[j] * H) + v);
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (p[j] < 0) continue;
        const uint32_t u[4] = {ld[j].x, ld[j].y, ld[j].z, ld[j].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float yv = __uint_as_float((i & 1) ? (u[i >> 1] & 0xffff0000u) : (u[i >> 1] << 16));
          float r = __fmul_rn(yv, w[j]);
          if (MODE == kAmax) {
            amax = fmaxf(amax, fabsf(r));
            continue;
          }
          if (FQ) r = fq_tbl[f32_to_e4m3(__fmul_rn(r, s))];
          acc[i] = __fadd_rn(acc[i], r);
        }
      }
      if (MODE == kAmax) continue;
      if (srow >= 0) {
        const uint4 sv = __ldg(reinterpret_cast<const uint4*>(shared_y + (size_t)srow * H) + v);
        const uint32_t u[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
          acc[i] = __fadd_rn(acc[i],
                             __uint_as_float((i & 1) ? (u[i >> 1] & 0xffff0000u) : (u[i >> 1] << 16)));
      }
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o[i] = (uint32_t)f32_to_bf16(acc[2 * i]) | ((uint32_t)f32_to_bf16(acc[2 * i + 1]) << 16);
      const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
      if (MODE == kWrite) {
        reinterpret_cast<uint4*>(out + (size_t)t * H)[v] = ov;
      } else {
        const uint4 ev = __ldg(reinterpret_cast<const uint4*>(expected + (size_t)t * H) + v);
        mismatch |= (ev.x != ov.x) | (ev.y != ov.y) | (ev.z != ov.z) | (ev.w != ov.w);
      }
    }
  }
  if (MODE == kVerify) {
    if (__ballot_sync(0xffffffffu, mismatch) && lane == 0) atomicOr(dev_status, MOE_DEV_VERIFY_MISMATCH);
  }
  if (MODE == kAmax) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    // non-negative floats order like their bit patterns as signed ints
    if (lane == 0 && amax > 0.0f) atomicMax(reinterpret_cast<int*>(amax_out), __float_as_int(amax));
  }
}

__global__ void fq_scale_kernel(const float* amax, float* scale, float top) {
  const float a = *amax;
  *scale = a > 0.0f ? __fdiv_rn(top, a) : 1.0f;
}

// ------------------------------------------------------------------ NVFP4 fake-quant
// The Mega-MoE page runs its combine quantiser with NVFP4 units as well as FP8 ones and
// leaves the format's arithmetic to that recipe; this is the two-level NVFP4 reading.
// Per 16 consecutive columns of a router-weighted row r (float32):
//   a = max |r|;  s_b = e4m3(fl32(fl32(a / 6) * g)) with g the per-tensor scale;
//   inv = fl32(g / s_b) (0 if s_b is 0);  d = fl32(s_b / g);
//   r' = fl32(e2m1(fl32(r * inv)) * d),
// e2m1 rounding to nearest even on the magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 and saturating.

// One warp per (token, column part) as in combine_kernel; a 16-column block is the two
// 8-column vectors of lanes 2m and 2m+1, which exchange their amax with one shuffle, so
// every lane runs the same iterations (parts hold an even number of vectors).
// K <= 8 (KMAX 8): capped at 64 registers so that 4 blocks (32 warps) share an SM, as the
// plain combine's; K > 8 keeps its 32-slot loads.
template <int KMAX, bool SPLIT>
__global__ void __launch_bounds__(256, KMAX <= 8 ? 4 : 1) combine_nvfp4_kernel(
    const uint16_t* __restrict__ y, const int32_t* __restrict__ inv_map, const float* __restrict__ topk_w, int T,
    int K, int H, const uint16_t* __restrict__ shared_y, const int32_t* __restrict__ shared_map,
    const float* __restrict__ g_scale, uint16_t* __restrict__ out, int splits) {
  const int lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int nvec = H / 8;
  const int per_part = SPLIT ? ((nvec + splits - 1) / splits + 1) & ~1 : nvec;
  const float g = *g_scale;
  // per block-scale code c: inv = fl32(g / decode(c)) (0 for a zero scale) and
  // d = fl32(decode(c) / g) -- the IEEE divisions each block would do, made once per code
  __shared__ float inv_tbl[256], d_tbl[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) {
    const float sd = e4m3_to_f32((uint8_t)i);
    inv_tbl[i] = sd > 0.0f ? __fdiv_rn(g, sd) : 0.0f;
    d_tbl[i] = __fdiv_rn(sd, g);
  }
  __syncthreads();
  const int n_items = SPLIT ? T * splits : T;
  for (int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < n_items; item += nw) {
    const int t = SPLIT ? item / splits : item;
    const int v_begin = SPLIT ? (item - t * splits) * per_part : 0;
    const int v_end = SPLIT ? min(nvec, v_begin + per_part) : nvec;
    if (v_begin >= v_end) continue;
    int my_p = -1;
    float my_w = 0.0f;
    if (lane < K) {
      my_p = inv_map[(size_t)t * K + lane];
      my_w = topk_w ? topk_w[(size_t)t * K + lane] : 1.0f;
    }
    const unsigned valid = __ballot_sync(0xffffffffu, lane < K && my_p >= 0);
    int srow = -1;
    if (valid && shared_y) srow = shared_map ? shared_map[t] : t;
    int p[KMAX];
    float w[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      p[j] = __shfl_sync(0xffffffffu, my_p, j);
      w[j] = __shfl_sync(0xffffffffu, my_w, j);
      if (j >= K) p[j] = -1;
    }
    for (int vb = v_begin; vb < v_end; vb += 32) {
      const int v = vb + lane;
      const bool act = v < v_end;     // the same for both lanes of a block (v_end is even)
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      uint4 ld[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        ld[j] = make_uint4(0u, 0u, 0u, 0u);
        if (p[j] >= 0 && act) ld[j] = __ldg(reinterpret_cast<const uint4*>(y + (size_t)p[j] * H) + v);
      }
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (p[j] < 0) continue;       // warp-uniform
        const uint32_t u[4] = {ld[j].x, ld[j].y, ld[j].z, ld[j].w};
        float r[8];
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float yv = __uint_as_float((i & 1) ? (u[i >> 1] & 0xffff0000u) : (u[i >> 1] << 16));
          r[i] = __fmul_rn(yv, w[j]);
          a = fmaxf(a, fabsf(r[i]));
        }
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        const uint8_t sc = f32_to_e4m3(__fmul_rn(__fdiv_rn(a, 6.0f), g));
        const float inv = inv_tbl[sc];
        const float d = d_tbl[sc];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          float q0, q1;
          e2m1_round2(__fmul_rn(r[i], inv), __fmul_rn(r[i + 1], inv), q0, q1);
          acc[i] = __fadd_rn(acc[i], __fmul_rn(q0, d));
          acc[i + 1] = __fadd_rn(acc[i + 1], __fmul_rn(q1, d));
        }
      }
      if (!act) continue;
      if (srow >= 0) {
        const uint4 sv = __ldg(reinterpret_cast<const uint4*>(shared_y + (size_t)srow * H) + v);
        const uint32_t u[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
          acc[i] = __fadd_rn(acc[i],
                             __uint_as_float((i & 1) ? (u[i >> 1] & 0xffff0000u) : (u[i >> 1] << 16)));
      }
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o[i] = (uint32_t)f32_to_bf16(acc[2 * i]) | ((uint32_t)f32_to_bf16(acc[2 * i + 1]) << 16);
      reinterpret_cast<uint4*>(out + (size_t)t * H)[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

template <int MODE>
moe_status_t launch_combine(const uint16_t* y, const int32_t* inv_map, const float* topk_w, int T, int K, int H,
                            const uint16_t* shared_y, const int32_t* shared_map, const float* fq_scale,
                            uint16_t* out, const uint16_t* expected, int32_t* dev_status, float* amax,
                            cudaStream_t s) {
  // split a token's columns over several warps when T warps cannot fill the GPU (64
  // resident warps per SM)
  const int target_warps = num_sms() * 64;
  const int splits = std::max(1, std::min(H / 8 / 32, target_warps / std::max(T, 1)));
  const long long items = (long long)T * splits;
  const int blocks = (int)std::min<long long>((items + 7) / 8, num_sms() * 16);
  const bool fq = fq_scale != nullptr && MODE != kAmax;
#define MOE_COMBINE_LAUNCH(FQV, KM, SP)                                                                 \
  combine_kernel<MODE, FQV, KM, SP><<<blocks, 256, 0, s>>>(y, inv_map, topk_w, T, K, H, shared_y, shared_map, \
                                                           fq_scale, out, expected, dev_status, amax, splits)
#define MOE_COMBINE_LAUNCH_K(FQV, SP) \
  if (K <= 8) MOE_COMBINE_LAUNCH(FQV, 8, SP); else MOE_COMBINE_LAUNCH(FQV, 32, SP);
  if (splits > 1) {
    if (fq) { MOE_COMBINE_LAUNCH_K(true, true) } else { MOE_COMBINE_LAUNCH_K(false, true) }
  } else {
    if (fq) { MOE_COMBINE_LAUNCH_K(true, false) } else { MOE_COMBINE_LAUNCH_K(false, false) }
  }
#undef MOE_COMBINE_LAUNCH_K
#undef MOE_COMBINE_LAUNCH
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

inline moe_status_t check_combine_args(const uint16_t* y, const int32_t* inv_map, const float* topk_w, int T,
                                       int K, int H, const uint16_t* shared_y) {
  if (T < 0 || K < 1 || K > kMaxTopK || H <= 0 || H % 128 != 0) return MOE_ERR_ARG;
  if (T > 0 && (!y || !inv_map)) return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(shared_y)) & 15) return MOE_ERR_ARG;
  return MOE_OK;
}

}  // namespace moe

extern "C" moe_status_t moe_combine(const uint16_t* y, const int32_t* inv_map, const float* topk_w, int T, int K,
                                    int H, const uint16_t* shared_y, const int32_t* shared_map,
                                    const float* fq_scale, uint16_t* out, void* stream) {
  using namespace moe;
  moe_status_t st = check_combine_args(y, inv_map, topk_w, T, K, H, shared_y);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!out || (reinterpret_cast<uintptr_t>(out) & 15)) return MOE_ERR_ARG;
  return launch_combine<kWrite>(y, inv_map, topk_w, T, K, H, shared_y, shared_map, fq_scale, out, nullptr,
                                nullptr, nullptr, as_stream(stream));
}

extern "C" moe_status_t moe_combine_verify(const uint16_t* y, const int32_t* inv_map, const float* topk_w, int T,
                                           int K, int H, const uint16_t* shared_y, const int32_t* shared_map,
                                           const float* fq_scale, const uint16_t* expected, int32_t* dev_status,
                                           void* stream) {
  using namespace moe;
  moe_status_t st = check_combine_args(y, inv_map, topk_w, T, K, H, shared_y);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!expected || !dev_status || (reinterpret_cast<uintptr_t>(expected) & 15)) return MOE_ERR_ARG;
  return launch_combine<kVerify>(y, inv_map, topk_w, T, K, H, shared_y, shared_map, fq_scale, nullptr, expected,
                                 dev_status, nullptr, as_stream(stream));
}

extern "C" moe_status_t moe_combine_amax(const uint16_t* y, const int32_t* inv_map, const float* topk_w, int T,
                                         int K, int H, float* amax, void* stream) {
  using namespace moe;
  moe_status_t st = check_combine_args(y, inv_map, topk_w, T, K, H, nullptr);
  if (st != MOE_OK) return st;
  if (!amax) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  return launch_combine<kAmax>(y, inv_map, topk_w, T, K, H, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                               amax, as_stream(stream));
}

extern "C" moe_status_t moe_fq_scale_from_amax(const float* amax, float* scale, void* stream) {
  using namespace moe;
  if (!amax || !scale) return MOE_ERR_ARG;
  fq_scale_kernel<<<1, 1, 0, as_stream(stream)>>>(amax, scale, 448.0f);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

extern "C" moe_status_t moe_fq4_scale_from_amax(const float* amax, float* scale, void* stream) {
  using namespace moe;
  if (!amax || !scale) return MOE_ERR_ARG;
  fq_scale_kernel<<<1, 1, 0, as_stream(stream)>>>(amax, scale, 2688.0f);   // 448 * 6
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

extern "C" moe_status_t moe_combine_nvfp4(const uint16_t* y, const int32_t* inv_map, const float* topk_w, int T,
                                          int K, int H, const uint16_t* shared_y, const int32_t* shared_map,
                                          const float* g_scale, uint16_t* out, void* stream) {
  using namespace moe;
  moe_status_t st = check_combine_args(y, inv_map, topk_w, T, K, H, shared_y);
  if (st != MOE_OK) return st;
  if (!g_scale) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!out || (reinterpret_cast<uintptr_t>(out) & 15)) return MOE_ERR_ARG;
  const int target_warps = num_sms() * 64;
  const int splits = std::max(1, std::min(H / 8 / 32, target_warps / std::max(T, 1)));
  const long long items = (long long)T * splits;
  const int blocks = (int)std::min<long long>((items + 7) / 8, num_sms() * 16);
  cudaStream_t s = as_stream(stream);
#define MOE_NVFP4_LAUNCH(KM, SP)                                                                         \
  combine_nvfp4_kernel<KM, SP><<<blocks, 256, 0, s>>>(y, inv_map, topk_w, T, K, H, shared_y, shared_map, \
                                                      g_scale, out, splits)
  if (splits > 1) {
    if (K <= 8) MOE_NVFP4_LAUNCH(8, true); else MOE_NVFP4_LAUNCH(32, true);
  } else {
    if (K <= 8) MOE_NVFP4_LAUNCH(8, false); else MOE_NVFP4_LAUNCH(32, false);
  }
#undef MOE_NVFP4_LAUNCH
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}
