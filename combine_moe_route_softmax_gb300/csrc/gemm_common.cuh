// Shared pieces of the tcgen05 grouped GEMM kernels (gemm.cu: one CTA per tile, behind
// every grouped-GEMM call and the layer; gemm2sm.cu: BF16 on CTA pairs with the 2-SM MMA,
// behind moe_grouped_gemm_pairs): tile constants, launch arguments, PTX wrappers, the unit
// decoder.  Internal header.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"


namespace moe {
namespace gg {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int KB_BYTES = 128;
constexpr int A_BYTES = BM * KB_BYTES;
constexpr int B_BYTES = BN * KB_BYTES;
constexpr int B_HALF = B_BYTES / 2;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr int MAX_SEG = kMaxExperts + 1;
constexpr unsigned long long TIMEOUT_NS = 2000000000ull;

// Per-warp shared-memory transpose of the BF16 epilogue: 32 rows x 64 bytes (four 16-byte
// chunks per row).  Chunk c of row r sits at chunk position c ^ ((r >> 1) & 3): a store of
// chunk c by 8 consecutive rows, and a load of 2 consecutive rows' 4 chunks, each touch 32
// distinct banks, so neither access conflicts.
constexpr int STAGE_OUT_PITCH = 64;
constexpr int STAGE_OUT_BYTES = 32 * STAGE_OUT_PITCH;
__device__ __forceinline__ int stage_out_off(int row, int chunk) {
  return row * STAGE_OUT_PITCH + ((chunk ^ ((row >> 1) & 3)) << 4);
}

constexpr int SMEM_MAX = 227 * 1024;
constexpr int NS = 32;   // rows of a segment computed on the streaming CTAs (at most)


struct Args {
  const int32_t* cu;        // cu_seqlens [nseg + 1], or masked_m [nseg] when max_tokens > 0
  int max_tokens;           // 0: contiguous segments; > 0: segment s owns rows [s*max_tokens, ...)
  int nseg;
  int rows_cap;
  int k_dim;
  int n_dim;
  int num_w;
  const float* a_scales;
  const float* w_scales;
  const float* wx_scales;
  void* out;
  float* out_scales;
  int32_t* dev_status;
  const float* row_scale;   // plain epilogue: out row r is multiplied by row_scale[r] (nullable)
  // fused combine (FUSE): out holds the BF16 expert rows; each token's output row is their
  // fixed-order sum, computed by the warp whose store completes the token's 128-column block
  const int32_t* src_row;   // row -> source index (t*K + k, or T*K + t for a shared row)
  const int32_t* inv_map;   // [T, K] slot -> row or -1
  const float* topk_w;      // [T, K] router weights, NULL for rows stored weighted
  const int32_t* shared_map;  // [T] token -> shared row or -1 (nullable)
  const float* fq_scale;    // combine fake-quant scale (nullable)
  uint16_t* comb_out;       // [T, n_dim] BF16
  int32_t* counters;        // [T, n_dim / 128], zero on entry, left zero
  int T, K;
  int stream;               // 1: segments of at most NS rows go to streaming CTAs
  int w_tiled;              // 1: weights in the tile layout of moe_pack_weights (single-CTA kernel)
  int common_off;           // shared-memory offset of the common tail
  unsigned long long timeout_ns;  // limit of each pipeline wait (TIMEOUT_NS; shorter only in tests)
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait (timeout_ns); false if the pipeline was aborted (by this wait timing out or
// another role).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* dev_status, unsigned long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (globaltimer() - t0 > timeout_ns) {
      *abort_flag = 1;
      if (dev_status) atomicOr(dev_status, MOE_DEV_PIPELINE_TIMEOUT);
      return false;
    }
  }
  return true;
}
// Bounded wait used while draining after an abort (ignores the abort flag).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > TIMEOUT_NS) return;
  }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// Prefetch of one box into L2 (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}
// With an L2 cache policy (createpolicy) attached to the copy.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
template <bool FP8>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  if (FP8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
  }
}
// 32 consecutive float32 columns of this warp's 32 TMEM lanes (one row per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 16 consecutive float32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// All `nthreads` threads of named barrier `id` arrive; true on every thread if any passed true.
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes,
// 8-row groups 1024 bytes apart (stride byte offset), start address in 16-byte units.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(1) << 16;             // leading byte offset (unused with 128B swizzle)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;     // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;             // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;             // 128-byte swizzle
  return d;
}
// Instruction descriptor: D float32, A/B K-major, N = BN, M = BM; A/B BF16 or E4M3.
template <bool FP8>
__host__ __device__ constexpr uint32_t instr_desc() {
  return (1u << 4) | ((FP8 ? 0u : 1u) << 7) | ((FP8 ? 0u : 1u) << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>(BM >> 4) << 24);
}
// BF16 x BF16 -> float32, M = 128 weight rows, N = NS token columns (streaming CTAs).
__host__ __device__ constexpr uint32_t instr_desc_stream() {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(NS >> 3) << 17) |
         (static_cast<uint32_t>(BM >> 4) << 24);
}

// SiLU with the fast exponential and divide: their relative error (a few 1e-6) is far
// below the BF16 or E4M3 rounding of h that follows; for g < -87 the denominator exceeds
// 2^126 and the quotient flushes to 0, the limit of g * sigmoid(g).
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// ------------------------------------------------------------- BF16 epilogue stores
// SwiGLU: this thread's 64 values of h (one row, 64 consecutive output columns) as BF16,
// 128 contiguous bytes at dst.
__device__ __forceinline__ void store_h_bf16(const float (&h)[64], uint16_t* dst) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = (uint32_t)f32_to_bf16(h[8 * v + 2 * j]) | ((uint32_t)f32_to_bf16(h[8 * v + 2 * j + 1]) << 16);
    d[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}
// Plain epilogue: the warp's 32 rows (lane = row) x 128 columns of acc as BF16 rows through
// the per-warp shared-memory transpose (buf_w, STAGE_OUT_BYTES): each lane holds one row,
// but a store instruction should cover whole sectors, so each 32-column chunk is written to
// shared memory row by row and read back as 8 rows x 64 contiguous bytes.  Rows
// [0, rows_here) of the warp are stored, row r at out + (row0 + r) * out_cols + col0.
__device__ __forceinline__ void store_rows_bf16(const float (&acc)[128], uint8_t* buf_w, int lane, int rows_here,
                                                uint16_t* out, int row0, int out_cols, int col0) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = (uint32_t)f32_to_bf16(acc[32 * c + 8 * v + 2 * j]) |
               ((uint32_t)f32_to_bf16(acc[32 * c + 8 * v + 2 * j + 1]) << 16);
      *reinterpret_cast<uint4*>(buf_w + stage_out_off(lane, v)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = (lane >> 2) + 8 * i;                 // row within the warp's 32
      const int ch = lane & 3;                           // 16-byte chunk of the row's 64 B
      const uint4 val = *reinterpret_cast<const uint4*>(buf_w + stage_out_off(r, ch));
      if (r < rows_here) {
        uint16_t* dst = out + (size_t)(row0 + r) * out_cols + col0 + 32 * c;
        reinterpret_cast<uint4*>(dst)[ch] = val;
      }
    }
    __syncwarp();
  }
}

struct Unit {
  int seg, row0, row_end, nt;
};
// Segment bounds kept in shared memory as bnd[]: contiguous segments [bnd[s], bnd[s+1]);
// batched segments [s*max_tokens, bnd[s]) (bnd[s] = the segment's end row).
__device__ __forceinline__ int seg_begin(const int* bnd, int s, int max_tokens) {
  return max_tokens > 0 ? s * max_tokens : bnd[s];
}
__device__ __forceinline__ int seg_end(const int* bnd, int s, int max_tokens) {
  return max_tokens > 0 ? bnd[s] : bnd[s + 1];
}
// Unit order within a segment: groups of `mgroup` M-tiles; inside a group, for each pair of
// N-tiles (one N-tile when the count is odd) every M-tile of the group in turn.  A round of
// the grid then holds a few weight tiles read by many M-tiles, so a large expert's weights
// cross HBM about once per group instead of once per round, while two consecutive units
// still share an M-tile (read from L2 by both).  mgroup = 0: M-tile-major order.
// Used for the BF16 gate/up (7168-deep K: a weight tile is 3.7 MB); the down projection's
// short units ran slower grouped (1.86 against 1.83 ms) and keep the M-tile-major order.
constexpr int MGROUP_GATE_UP = 32;
__device__ __forceinline__ Unit decode_unit(int u, int n_tiles, const int* cu, const int* prefix, int nseg,
                                            int max_tokens, int mgroup) {
  Unit w;
  const int mt = u / n_tiles;
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= mt)
      lo = mid;
    else
      hi = mid - 1;
  }
  w.seg = lo;
  int lm;
  if (mgroup == 0) {
    lm = mt - prefix[lo];
    w.nt = u - mt * n_tiles;
  } else {
    const int m = prefix[lo + 1] - prefix[lo];
    const int l = u - prefix[lo] * n_tiles;
    const int g = l / (mgroup * n_tiles);
    const int gs = min(mgroup, m - g * mgroup);
    const int r = l - g * mgroup * n_tiles;
    const int npw = (n_tiles & 1) ? 1 : 2;
    const int chunk = npw * gs;
    const int np = r / chunk;
    const int rr = r - np * chunk;
    lm = g * mgroup + rr / npw;
    w.nt = np * npw + (rr - (rr / npw) * npw);
  }
  w.row0 = seg_begin(cu, lo, max_tokens) + lm * BM;
  w.row_end = seg_end(cu, lo, max_tokens);
  return w;
}

// ---------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();
// rows x inner-elements matrix, box = box_rows rows x 128 bytes, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, bool fp8, uint64_t inner, uint64_t rows, uint32_t box_rows = 128);
// BF16 grouped GEMM on CTA pairs (gemm2sm.cu); args filled except stream / common_off.
moe_status_t launch_2sm(const void* a, int rows_cap, int k_dim, int n_dim, const void* w, int num_w,
                        const void* w_extra, bool swiglu, const Args& args, bool stream_ok, cudaStream_t s);

}  // namespace gg
}  // namespace moe
