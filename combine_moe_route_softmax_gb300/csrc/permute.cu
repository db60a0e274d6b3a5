// Permute (dispatch into the expert-major layout): stable counting sort of the valid
// (token, slot) pairs by expert id, then a gather of each row's token activations.
//
// MoonEP page: after dispatch the rows are laid out expert by expert ([NvS, H]) with
// cu_seqlens marking the segments, and the experts run as a grouped GEMM over them.
// Permute-scratch page: the scratch is sized from the inputs actually received and
// carries index data only.  DeepEP page: the low-latency dispatch accepts BF16 tokens and
// can quantise them to FP8 itself, shipping codes plus scales that the receiver
// dequantises -- here the 1x128 quantisation is fused into the row gather.
//
// Four launches, none of which waits on another block:
//   count   per-block per-segment histograms -> counts[seg][block]   (reads T*K*4 B)
//   scan    one block per segment: exclusive prefix over that segment's blocks; the
//           last block to finish (an atomic ticket, no waiting) scans the segment totals
//           into cu_seqlens
//   scatter per-block: per-warp histograms, a warp-level scan, then an ordered walk with
//           __match_any_sync ranks -> src_row / inv_map / shared_map (stable by slot)
//           (batched layout: the row of rank r in segment e goes to e*max_tokens + r,
//           ranks past max_tokens are dropped, and masked_m[e] = min(count, max_tokens))
//   gather  source-ordered: each token's row is read once and written to every row that
//           holds it (the token's slots and its shared row): BF16 rows through TMA bulk
//           copies staged in shared memory, E4M3 codes + 1x128 scales (or dispatch
//           fake-quantised rows) through 16-byte vector loads and stores.  HBM-bound:
//           T_valid*H*2 read + N*H*(2 | 1 + 4/128) written.
#include "common.cuh"

namespace moe {

constexpr int kPermThreads = 256;
constexpr int kPermWarps = kPermThreads / 32;
constexpr int kChunkTok = 64;                 // tokens per count/scatter block
constexpr int kTokPerWarp = kChunkTok / kPermWarps;

__device__ __forceinline__ bool valid_id(int e, int E) { return e >= 0 && e < E; }

__global__ void __launch_bounds__(kPermThreads) permute_count_kernel(const int32_t* __restrict__ idx, int T,
                                                                     int K, int E, int with_shared,
                                                                     int32_t* __restrict__ counts,
                                                                     int32_t* __restrict__ ticket,
                                                                     int32_t* dev_status,
                                                                     int32_t* __restrict__ zero_buf,
                                                                     int zero_per_token) {
  extern __shared__ int hist[];
  const int nseg = E + with_shared;
  for (int i = threadIdx.x; i < nseg; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * kChunkTok;
  const int t1 = min(T, t0 + kChunkTok);
  bool bad = false;
  for (int s = t0 * K + threadIdx.x; s < t1 * K; s += blockDim.x) {
    const int e = idx[s];
    if (valid_id(e, E))
      atomicAdd(&hist[e], 1);
    else if (e != -1)
      bad = true;
  }
  if (with_shared) {
    for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
      bool any = false;
      for (int k = 0; k < K; ++k) any |= valid_id(idx[(size_t)t * K + k], E);
      if (any) atomicAdd(&hist[E], 1);
    }
  }
  if (bad && dev_status) atomicOr(dev_status, MOE_DEV_BAD_EXPERT);
  if (blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0;
  if (zero_buf) {
    // per-token counters of a later fused combine, cleared for this block's tokens
    for (int i = threadIdx.x; i < (t1 - t0) * zero_per_token; i += blockDim.x)
      zero_buf[(size_t)t0 * zero_per_token + i] = 0;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nseg; i += blockDim.x) counts[(size_t)i * gridDim.x + blockIdx.x] = hist[i];
}

// Exclusive scan of v over the block's threads; returns this thread's exclusive prefix
// and (in *total) the block's sum.  blockDim.x == 256.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += u;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int ws = lane < 8 ? warp_sums[lane] : 0;
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, ws, off);
      if (lane >= off) ws += u;
    }
    if (lane < 8) warp_sums[lane] = ws;  // inclusive over warps
  }
  __syncthreads();
  const int excl = incl - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  *total = warp_sums[7];
  __syncthreads();
  return excl;
}

// One 256-thread block per segment e: counts[e][b] -> exclusive prefix over the blocks b
// (the row offset of block b's rows within segment e); seg_total[e] = segment size.  The
// last block to take a ticket scans the totals into cu_seqlens (cu[0] = 0) and resets the
// ticket.  No block ever waits for another.
__global__ void __launch_bounds__(256) permute_scan_kernel(int32_t* __restrict__ counts, int nblk, int nseg,
                                                           int32_t* __restrict__ seg_total,
                                                           int32_t* __restrict__ ticket,
                                                           int32_t* __restrict__ cu_seqlens) {
  __shared__ int warp_sums[8];
  __shared__ int last;
  const int e = blockIdx.x;
  int32_t* row = counts + (size_t)e * nblk;
  int running = 0;
  for (int base = 0; base < nblk; base += 256) {
    const int b = base + threadIdx.x;
    const int v = b < nblk ? row[b] : 0;
    int tot;
    const int ex = block_exclusive_scan(v, warp_sums, &tot);
    if (b < nblk) row[b] = running + ex;
    running += tot;
  }
  if (threadIdx.x == 0) {
    seg_total[e] = running;
    __threadfence();
    last = atomicAdd(ticket, 1) == nseg - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  running = 0;
  for (int base = 0; base < nseg; base += 256) {
    const int i = base + threadIdx.x;
    const int v = i < nseg ? __ldcg(seg_total + i) : 0;
    int tot;
    const int ex = block_exclusive_scan(v, warp_sums, &tot);
    if (i < nseg) cu_seqlens[i] = running + ex;
    running += tot;
  }
  if (threadIdx.x == 0) {
    cu_seqlens[nseg] = running;
    *ticket = 0;
  }
}

__global__ void __launch_bounds__(kPermThreads) permute_scatter_kernel(
    const int32_t* __restrict__ idx, int T, int K, int E, int with_shared, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ cu_seqlens, int cap, int32_t* __restrict__ src_row, int32_t* __restrict__ inv_map,
    int32_t* __restrict__ shared_map, const float* __restrict__ topk_w, float* __restrict__ row_w, int max_tokens,
    int32_t* __restrict__ masked_m, int32_t* dev_status) {
  extern __shared__ int whist[];  // [kPermWarps][nseg]
  const int nseg = E + with_shared;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kPermWarps * nseg; i += blockDim.x) whist[i] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * kChunkTok;
  const int wt0 = min(T, t0 + warp * kTokPerWarp);
  const int wt1 = min(T, wt0 + kTokPerWarp);
  const int ws0 = wt0 * K, ws1 = wt1 * K;
  int* my = whist + warp * nseg;
  // 1. per-warp histogram
  for (int s = ws0 + lane; s < ws1; s += 32) {
    const int e = idx[s];
    if (valid_id(e, E)) atomicAdd(&my[e], 1);
  }
  if (with_shared) {
    for (int t = wt0 + lane; t < wt1; t += 32) {
      bool any = false;
      for (int k = 0; k < K; ++k) any |= valid_id(idx[(size_t)t * K + k], E);
      if (any) atomicAdd(&my[E], 1);
    }
  }
  __syncthreads();
  // 2. each warp's starting row per segment = block offset + earlier warps' counts
  // (batched layout: rows counted from the segment's block e*max_tokens)
  const bool batched = max_tokens > 0;
  for (int e = threadIdx.x; e < nseg; e += blockDim.x) {
    int run = (batched ? e * max_tokens : cu_seqlens[e]) + offsets[(size_t)e * gridDim.x + blockIdx.x];
    for (int w = 0; w < kPermWarps; ++w) {
      const int c = whist[w * nseg + e];
      whist[w * nseg + e] = run;
      run += c;
    }
  }
  __syncthreads();
  // 3. ordered walk: lanes holding the same expert rank themselves by lane order
  for (int base = ws0; base < ws1; base += 32) {
    const int s = base + lane;
    const bool inr = s < ws1;
    const int e = inr ? idx[s] : -1;
    const bool ok = inr && valid_id(e, E);
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
    int rank = 0;
    if (ok) {
      rank = __popc(peers & lanemask_lt());
      const int pos = my[e] + rank;
      if (batched && pos - e * max_tokens >= max_tokens) {
        inv_map[s] = -1;   // past the segment's block: dropped (flagged below, per segment)
      } else {
        src_row[pos] = s;
        if (row_w) row_w[pos] = topk_w[s];
        inv_map[s] = pos;
      }
    } else if (inr) {
      inv_map[s] = -1;
    }
    __syncwarp();
    if (ok && rank == 0) my[e] += __popc(peers);
    __syncwarp();
  }
  if (with_shared) {
    for (int tb = wt0; tb < wt1; tb += 32) {
      const int t = tb + lane;
      const bool inr = t < wt1;
      bool any = false;
      if (inr)
        for (int k = 0; k < K; ++k) any |= valid_id(idx[(size_t)t * K + k], E);
      const unsigned ball = __ballot_sync(0xffffffffu, any);
      if (any) {
        const int pos = my[E] + __popc(ball & lanemask_lt());
        if (batched && pos - E * max_tokens >= max_tokens) {
          shared_map[t] = -1;
        } else {
          src_row[pos] = T * K + t;
          if (row_w) row_w[pos] = 1.0f;
          shared_map[t] = pos;
        }
      } else if (inr) {
        shared_map[t] = -1;
      }
      __syncwarp();
      if (lane == 0) my[E] += __popc(ball);
      __syncwarp();
    }
  }
  if (!batched) {
    // rows past the last one: -1
    const int total = cu_seqlens[nseg];
    for (int p = total + blockIdx.x * blockDim.x + threadIdx.x; p < cap; p += gridDim.x * blockDim.x)
      src_row[p] = -1;
    return;
  }
  // batched: masked_m, the overflow flag, and -1 in every row of a block past its masked_m
  // (disjoint from the rows written above, so no ordering between blocks is needed)
  if (blockIdx.x == 0) {
    bool over = false;
    for (int e = threadIdx.x; e < nseg; e += blockDim.x) {
      const int c = cu_seqlens[e + 1] - cu_seqlens[e];
      masked_m[e] = min(c, max_tokens);
      over |= c > max_tokens;
    }
    if (over && dev_status) atomicOr(dev_status, MOE_DEV_OVERFLOW);
  }
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < cap; p += gridDim.x * blockDim.x) {
    const int e = p / max_tokens;
    if (p - e * max_tokens >= cu_seqlens[e + 1] - cu_seqlens[e]) src_row[p] = -1;
  }
}

// Destination rows of token t: its valid slots' rows (inv_map) and its shared row.  Lane
// k < K holds the row of slot k, lane K the shared row (or -1).
__device__ __forceinline__ int token_dest(const int32_t* __restrict__ inv_map, const int32_t* __restrict__ shared_map,
                                          int t, int K, int lane) {
  if (lane < K) return inv_map[(size_t)t * K + lane];
  if (lane == K && shared_map) return shared_map[t];
  return -1;
}

// Dispatch fake-quant of 8 BF16 values: bf16(e4m3(x * s) / s), float32 steps; the division
// of each E4M3 code by s comes from a table made once per block (tbl[c] = decode(c) / s).
__device__ __forceinline__ uint4 qdq8(const uint4 u, float s, const float* tbl) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xffff0000u);
    const float ql = tbl[f32_to_e4m3(__fmul_rn(lo, s))];
    const float qh = tbl[f32_to_e4m3(__fmul_rn(hi, s))];
    o[i] = (uint32_t)f32_to_bf16(ql) | ((uint32_t)f32_to_bf16(qh) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Dispatch fake-quant of 8 BF16 values in NVFP4 (the page's other dispatch unit): the
// 16-column block is these 8 and the 8 of the partner lane (lane ^ 1), whose amax arrives by
// shuffle (every lane of the warp calls this), then as the combine's NVFP4 step --
// s_b = e4m3(fl32(fl32(a / 6) * g)), q = e2m1(fl32(x * g / s_b)), fl32(q * s_b / g) -- with
// g / s_b and s_b / g from per-code tables, and the result rounded to BF16.
__device__ __forceinline__ uint4 qdq8_nvfp4(const uint4 u, float g, const float* inv_tbl, const float* d_tbl) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float v[8];
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    a = fmaxf(a, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
  }
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  const uint8_t sc = f32_to_e4m3(__fmul_rn(__fdiv_rn(a, 6.0f), g));
  const float inv = inv_tbl[sc], d = d_tbl[sc];
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float q0, q1;
    e2m1_round2(__fmul_rn(v[2 * i], inv), __fmul_rn(v[2 * i + 1], inv), q0, q1);
    o[i] = (uint32_t)f32_to_bf16(__fmul_rn(q0, d)) | ((uint32_t)f32_to_bf16(__fmul_rn(q1, d)) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Source-ordered gather: one warp per token, the row read once in chunks of 4 16-byte
// vectors per lane and written to each destination row.  With a dispatch scale (DQ 1:
// E4M3, 2: NVFP4), the routed destinations get the fake-quantised row and the shared row
// the original.
// With few tokens (decode) a token's columns are split over `splits` warps, each taking
// a run of whole 128-vector groups, so that the GPU has enough warps in flight.
template <int DQ>
__global__ void __launch_bounds__(256) permute_gather_bf16_kernel(const uint16_t* __restrict__ x, int T, int K,
                                                                  int H, const int32_t* __restrict__ inv_map,
                                                                  const int32_t* __restrict__ shared_map,
                                                                  const float* __restrict__ dq_scale,
                                                                  uint16_t* __restrict__ xp, int splits) {
  const int lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int nvec = H / 8;
  const int per_part = ((nvec + 127) / 128 + splits - 1) / splits * 128;   // vectors, whole groups
  const int ndst = K + 1;
  const float s = DQ ? *dq_scale : 1.0f;
  __shared__ float dq_tbl[DQ == 1 ? 256 : 1];
  __shared__ float inv_tbl[DQ == 2 ? 256 : 1], d_tbl[DQ == 2 ? 256 : 1];
  if (DQ == 1) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) dq_tbl[i] = __fdiv_rn(e4m3_to_f32((uint8_t)i), s);
    __syncthreads();
  }
  if (DQ == 2) {
    // per block-scale code: g / decode(code) (0 for a zero scale) and decode(code) / g
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
      const float sd = e4m3_to_f32((uint8_t)i);
      inv_tbl[i] = sd > 0.0f ? __fdiv_rn(s, sd) : 0.0f;
      d_tbl[i] = __fdiv_rn(sd, s);
    }
    __syncthreads();
  }
  for (int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < T * splits; item += nw) {
    const int t = item / splits;
    const int v_begin = (item - t * splits) * per_part;
    const int v_end = min(nvec, v_begin + per_part);
    const int my_dst = token_dest(inv_map, shared_map, t, K, lane);
    const unsigned live = __ballot_sync(0xffffffffu, lane < ndst && my_dst >= 0);
    if (!live) continue;                      // padding token: nothing to copy
    const uint4* in = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    for (int v0 = v_begin; v0 < v_end; v0 += 128) {
      uint4 r[4], q[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = v0 + lane + 32 * j;
        r[j] = make_uint4(0u, 0u, 0u, 0u);
        if (v < v_end) {
          r[j] = __ldg(in + v);
          if (DQ == 1) q[j] = qdq8(r[j], s, dq_tbl);
        }
        // NVFP4: every lane takes part in the block's amax shuffle; a lane past v_end holds
        // zeros, and so does its partner (parts hold whole 128-vector groups, v_end is even)
        if (DQ == 2) q[j] = qdq8_nvfp4(r[j], s, inv_tbl, d_tbl);
      }
      unsigned m = live;
      while (m) {
        const int d = __ffs(m) - 1;
        m &= m - 1;
        const int row = __shfl_sync(0xffffffffu, my_dst, d);
        const bool routed = d < K;
        uint4* o = reinterpret_cast<uint4*>(xp + (size_t)row * H);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int v = v0 + lane + 32 * j;
          if (v < v_end) o[v] = (DQ != 0 && routed) ? q[j] : r[j];
        }
      }
    }
  }
}

// ------------------------------------------------------- TMA-staged gather (BF16 rows)
// One bulk copy (cp.async.bulk) brings a token's row into shared memory; one bulk store per
// destination row writes it out as a single contiguous transfer.  Each warp runs a two-deep
// pipeline (the next token's row loads while the current one is stored); lane 0 issues the
// copies, the warp shares the destination rows.  Waits on the load barriers are bounded
// (2 s of globaltimer): on expiry the warp sets MOE_DEV_PIPELINE_TIMEOUT, waits (bounded)
// for its load in flight and stops.
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t smem_u32addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void bulk_row_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void bulk_row_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool bulk_bar_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = gtimer();
  for (;;) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if (gtimer() - t0 > 2000000000ull) return false;
  }
}

__global__ void __launch_bounds__(256) permute_gather_bf16_bulk_kernel(const uint16_t* __restrict__ x, int T, int K,
                                                                       int H, const int32_t* __restrict__ inv_map,
                                                                       const int32_t* __restrict__ shared_map,
                                                                       uint16_t* __restrict__ xp,
                                                                       int32_t* dev_status) {
  extern __shared__ __align__(128) uint8_t gsm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const uint32_t row_bytes = static_cast<uint32_t>(H) * 2;
  const uint32_t buf_stride = (row_bytes + 127) / 128 * 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gsm);                       // [nwarps][2]
  uint8_t* bufs = gsm + 128 + static_cast<size_t>(warp) * 2 * buf_stride;  // this warp's two rows
  const uint32_t bar0 = smem_u32addr(bars + 2 * warp);
  const uint32_t buf0 = smem_u32addr(bufs);
  if (lane == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  const int ndst = K + 1;
  const int nw = gridDim.x * nwarps;
  // the next token (stride nw) that has a row to write, or T
  auto next_live = [&](int t) {
    for (; t < T; t += nw) {
      const int d = token_dest(inv_map, shared_map, t, K, lane);
      if (__ballot_sync(0xffffffffu, lane < ndst && d >= 0)) return t;
    }
    return T;
  };
  int cur = next_live(blockIdx.x * nwarps + warp);
  int b = 0;
  uint32_t phases = 0;              // bit i: parity of buffer i's next load
  bool loading_next = false;        // a load into buffer b ^ 1 is in flight
  if (lane == 0 && cur < T) bulk_row_load(buf0, x + (size_t)cur * H, row_bytes, bar0);
  while (cur < T) {
    const int nxt = next_live(cur + nw);
    const int my_dst = token_dest(inv_map, shared_map, cur, K, lane);
    const unsigned live = __ballot_sync(0xffffffffu, lane < ndst && my_dst >= 0);
    const uint32_t nb = static_cast<uint32_t>(b ^ 1);
    if (lane == 0 && nxt < T) {
      // the stores of the token before `cur` read buffer nb: let them finish reading
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      bulk_row_load(buf0 + nb * buf_stride, x + (size_t)nxt * H, row_bytes, bar0 + 8 * nb);
    }
    loading_next = nxt < T;
    bool ok = true;
    if (lane == 0) ok = bulk_bar_wait(bar0 + 8 * b, (phases >> b) & 1u);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) {
        if (dev_status) atomicOr(dev_status, MOE_DEV_PIPELINE_TIMEOUT);
        if (loading_next) bulk_bar_wait(bar0 + 8 * nb, (phases >> nb) & 1u);
      }
      break;
    }
    phases ^= 1u << b;
    unsigned m = live;
    while (m) {
      const int d = __ffs(m) - 1;
      m &= m - 1;
      const int row = __shfl_sync(0xffffffffu, my_dst, d);
      if (lane == 0) bulk_row_store(xp + (size_t)row * H, buf0 + b * buf_stride, row_bytes);
    }
    if (lane == 0) asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    cur = nxt;
    b = static_cast<int>(nb);
  }
  // every store has been performed (and has read its row) before the warp leaves
  if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  __syncwarp();
}

// 1x128 quantisation of 8 elements per lane (a half-warp covers one 128-block): returns
// the 8 codes packed in a uint2 and the block's scale.  Every lane of the warp calls it.
__device__ __forceinline__ uint2 quant8(const uint4 u, bool live, float* scale) {
  float f[8];
  float amax = 0.0f;
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
  if (live) {
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float s = block_scale(amax);
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) lo |= (uint32_t)f32_to_e4m3(__fdiv_rn(f[i], s)) << (8 * i);
#pragma unroll
  for (int i = 0; i < 4; ++i) hi |= (uint32_t)f32_to_e4m3(__fdiv_rn(f[4 + i], s)) << (8 * i);
  *scale = s;
  return make_uint2(lo, hi);
}

// Source-ordered gather with the 1x128 E4M3 quantisation: each token is quantised once and
// its codes and scales written to every destination row.
__global__ void __launch_bounds__(256) permute_gather_e4m3_kernel(const uint16_t* __restrict__ x, int T, int K,
                                                                  int H, const int32_t* __restrict__ inv_map,
                                                                  const int32_t* __restrict__ shared_map,
                                                                  uint8_t* __restrict__ xp,
                                                                  float* __restrict__ xp_scales, int splits) {
  const int lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int nvec = H / 8;
  const int nblk = H / 128;
  // parts of whole 32-vector groups (two 1x128 blocks), so each half-warp keeps one block
  const int per_part = ((nvec + 31) / 32 + splits - 1) / splits * 32;
  const int ndst = K + 1;
  for (int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < T * splits; item += nw) {
    const int t = item / splits;
    const int v_begin = (item - t * splits) * per_part;
    const int v_end = min(nvec, v_begin + per_part);
    const int my_dst = token_dest(inv_map, shared_map, t, K, lane);
    const unsigned live = __ballot_sync(0xffffffffu, lane < ndst && my_dst >= 0);
    if (!live) continue;
    const uint4* in = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    for (int v0 = v_begin; v0 < v_end; v0 += 32) {
      const int v = v0 + lane;
      const bool ok = v < v_end;
      const uint4 u = ok ? __ldg(in + v) : make_uint4(0, 0, 0, 0);
      float s;
      const uint2 q = quant8(u, ok, &s);
      unsigned m = live;
      while (m) {
        const int d = __ffs(m) - 1;
        m &= m - 1;
        const int row = __shfl_sync(0xffffffffu, my_dst, d);
        if (ok) {
          reinterpret_cast<uint2*>(xp + (size_t)row * H)[v] = q;
          if ((lane & 15) == 0) xp_scales[(size_t)row * nblk + v / 16] = s;
        }
      }
    }
  }
}

__global__ void __launch_bounds__(256) quant_act_kernel(const uint16_t* __restrict__ x, int rows, int cols,
                                                        uint8_t* __restrict__ q, float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int nvec = cols / 8;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nw) {
    const uint4* in = reinterpret_cast<const uint4*>(x + (size_t)r * cols);
    for (int v0 = 0; v0 < nvec; v0 += 32) {
      const int v = v0 + lane;
      const bool ok = v < nvec;
      float s;
      const uint2 c = quant8(ok ? __ldg(in + v) : make_uint4(0, 0, 0, 0), ok, &s);
      if (ok) {
        reinterpret_cast<uint2*>(q + (size_t)r * cols)[v] = c;
        if ((lane & 15) == 0) scales[(size_t)r * (cols / 128) + v / 16] = s;
      }
    }
  }
}

inline int perm_blocks(int T) { return (T + kChunkTok - 1) / kChunkTok; }

// Index scratch: counts [nseg][nblk] | segment totals [nseg] | ticket (256-byte regions).
struct ScratchLayout {
  size_t counts, seg_total, ticket, total;
};
inline ScratchLayout scratch_layout(size_t nblk, size_t nseg) {
  auto a = [](size_t x) { return (x + 255) / 256 * 256; };
  ScratchLayout l;
  l.counts = 0;
  l.seg_total = a(nblk * nseg * sizeof(int32_t));
  l.ticket = l.seg_total + a(nseg * sizeof(int32_t));
  l.total = l.ticket + 256;
  return l;
}

}  // namespace moe

extern "C" size_t moe_permute_workspace_bytes(int T, int K, int E, int with_shared) {
  using namespace moe;
  if (T < 0 || K < 1 || E < 1 || E > kMaxExperts) return 0;
  const size_t nseg = (size_t)E + (with_shared ? 1 : 0);
  return scratch_layout(perm_blocks(T), nseg).total;
}

extern "C" size_t moe_permute_batched_workspace_bytes(int T, int K, int E, int with_shared) {
  // the contiguous scratch plus the segments' cu_seqlens, which the batched layout keeps
  // internal (its callers get masked_m)
  const size_t b = moe_permute_workspace_bytes(T, K, E, with_shared);
  if (b == 0) return 0;
  const size_t nseg = (size_t)E + (with_shared ? 1 : 0);
  return b + (nseg + 1) * sizeof(int32_t) + 255 - ((nseg + 1) * sizeof(int32_t) + 255) % 256;
}

namespace moe {
moe_status_t permute_impl(const int32_t* topk_idx, int T, int K, int E, int with_shared, const uint16_t* x,
                          int H, moe_dtype_t out_dtype, void* xp, float* xp_scales, int32_t* cu_seqlens,
                          int32_t* src_row, int32_t* inv_map, int32_t* shared_map, void* ws, size_t ws_bytes,
                          int32_t* dev_status, const float* dq_scale, const float* topk_w, float* row_w,
                          int max_tokens, int32_t* masked_m, void* stream, int32_t* zero_buf,
                          int zero_per_token, int dq_format){
  if (T < 0 || K < 1 || K > kMaxTopK || E < 1 || E > kMaxExperts || H <= 0 || H % 128 != 0) return MOE_ERR_ARG;
  if (with_shared != 0 && with_shared != 1) return MOE_ERR_ARG;
  if (out_dtype != MOE_BF16 && out_dtype != MOE_E4M3) return MOE_ERR_ARG;
  const bool batched = max_tokens != 0;
  const int nseg = E + with_shared;
  if (batched) {
    if (max_tokens < 0 || (size_t)nseg * max_tokens > 0x7fffffffull || !masked_m) return MOE_ERR_ARG;
  } else if (!cu_seqlens) {
    return MOE_ERR_ARG;
  }
  cudaStream_t s = as_stream(stream);
  if (T == 0) {
    int32_t* z = batched ? masked_m : cu_seqlens;
    if (cudaMemsetAsync(z, 0, sizeof(int32_t) * (batched ? nseg : nseg + 1), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (batched && src_row &&
        cudaMemsetAsync(src_row, 0xff, sizeof(int32_t) * (size_t)nseg * max_tokens, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  if (!topk_idx || !x || !xp || !src_row || !inv_map || (with_shared && !shared_map)) return MOE_ERR_ARG;
  if (out_dtype == MOE_E4M3 && !xp_scales) return MOE_ERR_ARG;
  if (dq_scale && out_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (dq_format != 0 && dq_format != 1) return MOE_ERR_ARG;
  if (row_w && !topk_w) return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(xp)) & 15) return MOE_ERR_ARG;
  if ((size_t)T * K + T > 0x7fffffffull) return MOE_ERR_ARG;
  const size_t need = batched ? moe_permute_batched_workspace_bytes(T, K, E, with_shared)
                              : moe_permute_workspace_bytes(T, K, E, with_shared);
  if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
  const int nblk = perm_blocks(T);
  const ScratchLayout lay = scratch_layout(nblk, nseg);
  uint8_t* base = static_cast<uint8_t*>(ws);
  int32_t* counts = reinterpret_cast<int32_t*>(base + lay.counts);
  int32_t* seg_total = reinterpret_cast<int32_t*>(base + lay.seg_total);
  int32_t* ticket = reinterpret_cast<int32_t*>(base + lay.ticket);
  if (batched) cu_seqlens = reinterpret_cast<int32_t*>(base + lay.total);
  const int cap = batched ? nseg * max_tokens : T * K + (with_shared ? T : 0);
  permute_count_kernel<<<nblk, kPermThreads, nseg * sizeof(int), s>>>(topk_idx, T, K, E, with_shared, counts,
                                                                        ticket, dev_status, zero_buf,
                                                                        zero_per_token);
  MOE_CHECK_LAUNCH();
  permute_scan_kernel<<<nseg, 256, 0, s>>>(counts, nblk, nseg, seg_total, ticket, cu_seqlens);
  MOE_CHECK_LAUNCH();
  const size_t scatter_smem = (size_t)kPermWarps * nseg * sizeof(int);
  // per-warp histograms of up to 1025 segments: 32.8 KB, under the 48 KB default limit
  static_assert(kPermWarps * (kMaxExperts + 1) * sizeof(int) <= 48 * 1024, "scatter histograms exceed 48 KB");
  permute_scatter_kernel<<<nblk, kPermThreads, scatter_smem, s>>>(topk_idx, T, K, E, with_shared, counts,
                                                                  cu_seqlens, cap, src_row, inv_map, shared_map,
                                                                  topk_w, row_w, batched ? max_tokens : 0,
                                                                  masked_m, dev_status);
  MOE_CHECK_LAUNCH();
  // column parts per token: enough warps to fill the GPU when tokens are few
  const int groups = out_dtype == MOE_BF16 ? (H / 8 + 127) / 128 : (H / 8 + 31) / 32;
  const int splits = std::max(1, std::min(groups, num_sms() * 64 / T));   // 64 resident warps per SM
  const long long items = (long long)T * splits;
  const int gblocks = (int)std::min<long long>((items + 7) / 8, num_sms() * 8);
  const int32_t* smap = with_shared ? shared_map : nullptr;
  // BF16 rows without dispatch fake-quant: TMA-staged gather, one 8-warp block per SM (two
  // row buffers per warp) when two rows per warp fit in shared memory
  const size_t row_buf = ((size_t)H * 2 + 127) / 128 * 128;
  const int bulk_warps = (int)std::min<size_t>(8, (232448 - 128) / (2 * row_buf));
  if (out_dtype == MOE_BF16 && !dq_scale && bulk_warps >= 1) {
    const size_t smem = 128 + (size_t)bulk_warps * 2 * row_buf;
    static std::atomic<unsigned long long> attr_done{0};
    if (!once_per_device(attr_done, [&] {
          return cudaFuncSetAttribute(permute_gather_bf16_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      232448) == cudaSuccess;
        }))
      return MOE_ERR_CUDA;
    const int blocks = std::max(1, std::min(num_sms(), (T + bulk_warps - 1) / bulk_warps));
    permute_gather_bf16_bulk_kernel<<<blocks, bulk_warps * 32, smem, s>>>(x, T, K, H, inv_map, smap,
                                                                          static_cast<uint16_t*>(xp), dev_status);
  } else if (out_dtype == MOE_BF16)
    if (dq_scale && dq_format == 1)
      permute_gather_bf16_kernel<2><<<gblocks, 256, 0, s>>>(x, T, K, H, inv_map, smap, dq_scale,
                                                            static_cast<uint16_t*>(xp), splits);
    else if (dq_scale)
      permute_gather_bf16_kernel<1><<<gblocks, 256, 0, s>>>(x, T, K, H, inv_map, smap, dq_scale,
                                                            static_cast<uint16_t*>(xp), splits);
    else
      permute_gather_bf16_kernel<0><<<gblocks, 256, 0, s>>>(x, T, K, H, inv_map, smap, nullptr,
                                                            static_cast<uint16_t*>(xp), splits);
  else
    permute_gather_e4m3_kernel<<<gblocks, 256, 0, s>>>(x, T, K, H, inv_map, smap, static_cast<uint8_t*>(xp),
                                                       xp_scales, splits);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}
}  // namespace moe

extern "C" moe_status_t moe_permute(const int32_t* topk_idx, int T, int K, int E, int with_shared,
                                    const uint16_t* x, int H, moe_dtype_t out_dtype, void* xp,
                                    float* xp_scales, int32_t* cu_seqlens, int32_t* src_row, int32_t* inv_map,
                                    int32_t* shared_map, void* ws, size_t ws_bytes, int32_t* dev_status,
                                    void* stream) {
  return moe::permute_impl(topk_idx, T, K, E, with_shared, x, H, out_dtype, xp, xp_scales, cu_seqlens, src_row,
                           inv_map, shared_map, ws, ws_bytes, dev_status, nullptr, nullptr, nullptr, 0, nullptr,
                           stream, nullptr, 0);
}

extern "C" moe_status_t moe_permute_ex(const int32_t* topk_idx, int T, int K, int E, int with_shared,
                                       const uint16_t* x, int H, moe_dtype_t out_dtype, void* xp,
                                       float* xp_scales, int32_t* cu_seqlens, int32_t* src_row, int32_t* inv_map,
                                       int32_t* shared_map, void* ws, size_t ws_bytes, int32_t* dev_status,
                                       const float* dispatch_scale, int dispatch_format, const float* topk_w,
                                       float* row_weights, void* stream) {
  return moe::permute_impl(topk_idx, T, K, E, with_shared, x, H, out_dtype, xp, xp_scales, cu_seqlens, src_row,
                           inv_map, shared_map, ws, ws_bytes, dev_status, dispatch_scale, topk_w, row_weights, 0,
                           nullptr, stream, nullptr, 0, dispatch_format);
}

extern "C" moe_status_t moe_permute_batched(const int32_t* topk_idx, int T, int K, int E, int with_shared,
                                            int max_tokens, const uint16_t* x, int H, moe_dtype_t out_dtype,
                                            void* xb, float* xb_scales, int32_t* masked_m, int32_t* src_row,
                                            int32_t* inv_map, int32_t* shared_map, void* ws, size_t ws_bytes,
                                            int32_t* dev_status, const float* dispatch_scale,
                                            int dispatch_format, const float* topk_w, float* row_weights,
                                            void* stream) {
  if (max_tokens < 1) return MOE_ERR_ARG;
  return moe::permute_impl(topk_idx, T, K, E, with_shared, x, H, out_dtype, xb, xb_scales, nullptr, src_row,
                           inv_map, shared_map, ws, ws_bytes, dev_status, dispatch_scale, topk_w, row_weights,
                           max_tokens, masked_m, stream, nullptr, 0, dispatch_format);
}

extern "C" moe_status_t moe_quantize_act_fp8(const uint16_t* x, int rows, int cols, uint8_t* q, float* scales,
                                             void* stream) {
  using namespace moe;
  if (rows < 0 || cols <= 0 || cols % 128 != 0) return MOE_ERR_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !q || !scales) return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(q) & 7)) return MOE_ERR_ARG;
  const int blocks = min((rows + 7) / 8, num_sms() * 8);
  quant_act_kernel<<<blocks, 256, 0, as_stream(stream)>>>(x, rows, cols, q, scales);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}
