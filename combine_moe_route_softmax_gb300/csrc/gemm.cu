// Grouped GEMM over the expert segments on the 5th-generation tensor cores (sm_103a):
// tcgen05.mma with accumulators in tensor memory (TMEM), operands staged in shared memory
// by TMA (cp.async.bulk.tensor, 128-byte swizzle), and a persistent
// per-expert tile scheduler that builds its tile list on the device from cu_seqlens, so
// the host never needs the segment lengths (no host sync; graph-capturable).
//
// MoonEP page: the experts run as three grouped matmuls (gate, up, down) over the
// cu_seqlens segments, and empty segments simply produce no tiles.  DeepEP page: gate and
// up are one fused weight with 2n rows; FP8 weights carry block_n x block_k scales.
//
// Tile: BM = 128 rows x BN = 256 weight rows x 128 bytes of K per pipeline stage
// (64 BF16 or 128 E4M3 elements), 4 stages (48 KB each); BF16 (not fused) units take two
// such M-tiles sharing the weight tile, 3 stages of 64 KB.  For SwiGLU the 256 weight rows
// of a tile are 128 gate rows and the matching 128 up rows, so one MMA with N = 256
// yields g and u for 128 output columns side by side in TMEM.
//
// Weights: row-major [num_w, n_dim, k_dim], where a 128-row x 128-byte box is 128 pieces a
// row apart, or the tile layout of moe_pack_weights (MOE_W_TILED), where it is 16
// contiguous KB; the kernel only addresses the box differently (wx / wy below).  The
// streamed weights of the short segments arrive faster from contiguous boxes (prefill
// gate/up 3.17-3.18 against 3.30-3.32 ms, same box).
//
// Two roles.  The MMA pipeline below takes every segment when streaming is off, and the
// segments of more than NS = 32 rows when it is on.  Streaming CTAs (the last ny CTAs of
// the grid, BF16 and not fused, when the launch has at least 16 units per CTA) take the
// segments of at most NS rows: such a segment is a weight stream, so its CTAs keep six
// 32 KB weight tiles in flight behind 4 KB token tiles and issue MMAs with the weights as
// the M = 128 operand and the segment's rows as N = NS, on two pipeline lanes (two TMA
// threads, two MMA threads, alternate K blocks).  Every CTA derives the same ny from the
// segment lengths and a per-unit cost model, so no host sync is needed.
//
// Warp roles of the MMA pipeline (320 threads, one CTA per SM):
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM allocator + MMA issuer (one lane)
//   warps 2..9  epilogue: warp w reads TMEM lanes 32*(w%4).. (its subpartition) and
//               half (w-2)/4 of the tile's columns.
// TMEM: 512 columns = two 256-column accumulator buffers, so the epilogue of one
// accumulation round overlaps the MMAs of the next.
//   BF16: one round per tile; the whole K loop accumulates in TMEM.  BF16 gate/up (not
//         fused) computes two M-tiles per unit instead, one accumulator each (below).
//   E4M3: one round per 128-wide K block: each block's partial product is scaled by its
//         activation scale (per row) and weight scale (per 128x128 block) and added into
//         float32 registers by the epilogue warps ("promotion"), since the scales are
//         float32 per 128 elements rather than a format the MMA applies itself.
//
// Warp roles of a streaming CTA: warps 0 and 6 TMA producers of pipeline lanes 0 and 1,
// warps 1 and 7 their MMA issuers (warp 1 also allocates TMEM), warps 2..5 epilogue.
//
// Every mbarrier wait is bounded (about 2 s of globaltimer); on expiry the CTA sets
// MOE_DEV_PIPELINE_TIMEOUT in the status word, every role leaves its loop, the producers
// wait (bounded) for their copies in flight, the MMA lanes wait (bounded) for their MMAs,
// and the TMEM is freed before the CTA exits.
#include "gemm_common.cuh"

namespace moe {
namespace gg {

constexpr int STAGES = 4;
constexpr int STAGE_TX = A_BYTES + B_BYTES;
// BF16 gate/up (not fused): an MMA-pipeline unit is two M-tiles of one segment sharing each
// weight tile (256 x 256 outputs, both 256-column accumulators in TMEM), so a K step moves
// 64 KB (two A tiles and one weight tile) for twice the work of a 48 KB single-tile step:
// a third fewer operand bytes per product, on a path whose tensor pipe waits about a fifth
// of its cycles for operand tiles.  Three 64 KB stages fill the same shared memory as four
// 48 KB ones.  The accumulators are not double-buffered; the epilogue frees the first one
// as soon as it has read it, and the next unit's MMAs into it start then (a single buffer
// cost 0.2-0.6 % on the one-tile path).
constexpr int STAGES_M2 = 3;
// Unit order of two-tile gate/up units: groups of 4 units (8 M-tiles), each pair of N-tiles
// visiting the group's units before the next pair, so a round of the grid covers every
// N-tile of a few M-tiles (their A rows read from L2 once per round) and the weights of a
// segment's N-tiles are shared by the round's groups.  Swept on the prefill routing (same
// box, three rounds): groups of 4 units 3.29-3.33 ms, 8: 3.30-3.35, 16 (the one-tile
// order's 32 M-tiles): 3.39-3.44, 32-64: 3.46-3.52.
constexpr int MGROUP_GATE_UP_M2 = 4;
// The down projection's two-tile units in groups of 8 the same way (its one-tile units kept
// the M-tile-major order, every N-tile of one M-tile before the next): 1.69-1.73 against
// 1.74-1.75 ms in same-box sweeps (groups of 2: 1.71-1.75, 16: 1.71-1.73).
constexpr int MGROUP_DOWN_M2 = 8;
constexpr int STAGE_M2_BYTES = 2 * A_BYTES + B_BYTES;   // 64 KB
static_assert(STAGES_M2 * STAGE_M2_BYTES == STAGES * (A_BYTES + B_BYTES), "same shared memory as the one-tile ring");

// Streamed segments (BF16, not fused): a segment of at most NS rows is computed by a
// streaming CTA with the weights as the MMA's M operand (two M = 128 halves of a 256-row
// weight tile) and the segment's rows as N = NS columns, through a deeper ring of
// weight-sized stages.  Such a segment's units are bound by streaming their weights, and
// one CTA keeps only four 32 KB weight tiles in flight behind 16 KB activation tiles that
// hold a few real rows; here it keeps six behind 4 KB token tiles.
constexpr int YSTAGES = 6;
constexpr int YT_BYTES = NS * KB_BYTES;
constexpr int YSTAGE_BYTES = B_BYTES + YT_BYTES;   // 36 KB, a multiple of 1024

struct SmemLayout {
  // MMA-pipeline CTAs
  static constexpr int a = 0;
  static constexpr int b = a + STAGES * A_BYTES;
  static constexpr int xch = b + STAGES * B_BYTES;            // float [2][128]
  static constexpr int stage_out = xch + 2 * 128 * 4;         // per epilogue warp: 32 x 64 B
  static constexpr int x_end = stage_out + EPI_WARPS * STAGE_OUT_BYTES;
  // streaming CTAs: YSTAGES x [256 weight rows | NS token rows]
  static constexpr int y_end = YSTAGES * YSTAGE_BYTES;
  // common tail at Args::common_off (after x_end, or after y_end when streaming is on):
  // barriers full[6], empty[6], tfull[2], tempty[2], drain[2]; TMEM slot; abort flag; role
  // split; then int cu[nseg + 1], prefix[nseg + 1], prefix_y[nseg + 1]
  static constexpr int n_bars = 2 * YSTAGES + 6;
  static constexpr int tmem_slot = n_bars * 8;
  static constexpr int abort_flag = tmem_slot + 4;
  static constexpr int costs = abort_flag + 4;                // float [2]
  static constexpr int arrays = 256;
  static size_t bytes(int common_off, int nseg) {
    return static_cast<size_t>(common_off) + arrays + ((3 * (nseg + 1) * 4 + 15) / 16) * 16 + 1024;  // + align slack
  }
};
static_assert(SmemLayout::costs + 8 <= SmemLayout::arrays, "common tail header");
static_assert(STAGES <= YSTAGES, "barrier slots");
// Streaming pipeline lanes: two for both GEMMs.  (With one M-tile per gate/up unit one lane
// was faster for gate/up: the faster weight stream took L2 and HBM bandwidth from that
// pipeline.  With two M-tiles per unit, which needs a third fewer operand bytes per product,
// two lanes are faster: gate/up 3.26-3.38 against 3.40-3.42 ms in same-box A/B runs.)
template <bool SWIGLU>
__host__ __device__ constexpr int y_lanes() { return 2; }
// Relative time of one unit (all units of a launch have the same K): an MMA-bound tile, a
// single-tile segment's tile on the MMA pipeline, a two-tile gate/up unit, and a streamed
// unit.  They set how many CTAs stream.  Measured per unit on the prefill expert mix with
// both roles running: a one-tile unit about 45 us on gate/up and 13 us on down, a streamed
// unit 37 and 11 us; the streamed cost is set above its measurement so that the streaming
// CTAs, which cannot hand work back, do not finish last.  The two-tile cost was swept:
// 92 gave 24 streaming CTAs and 40 rounds of gate/up units on the other 128 (gate/up
// 3.26-3.38 ms), 84-88 gave 25-26 streaming CTAs and 41 rounds (3.51-3.59 ms).
constexpr float COST_MMA = 46.0f, COST_SINGLE = 61.0f, COST_STREAM = 42.0f;
constexpr float COST_MMA2 = 92.0f;
// Streaming CTAs: warps 0 and Y_PRODUCER1 load the ring, warps 1 and Y_ISSUER1 issue the
// MMAs (one pair per pipeline lane), warps 2..5 are the epilogue (one unit streams for tens
// of microseconds; its epilogue is short).
constexpr int Y_EPI_WARPS = 4;
constexpr int Y_PRODUCER1 = 2 + Y_EPI_WARPS, Y_ISSUER1 = Y_PRODUCER1 + 1;  // lane 1 of the streaming pipeline
static_assert(Y_ISSUER1 < THREADS / 32, "streaming warps");
// A streamed weight tile is read once: its copies carry an L2 evict-first policy, so the
// streaming CTAs' gigabytes do not push out the weight tiles that the MMA pipeline's
// M-tiles of one segment share through L2.
constexpr bool STREAM_EVICT_FIRST = true;

// ----------------------------------------------------------------- fused combine
// Columns [col, col + 128) of token t's output: the combine's arithmetic on the stored BF16
// rows -- slots in ascending order, r = float(y) * w (float32 product), optional E4M3 QDQ,
// float32 sum from +0 without FMA, the shared row last (only for a token with a routed
// row), one BF16 rounding.  The whole warp works on the block: lane l owns 4 columns.  Rows
// are read through L2 (__ldcg): other SMs wrote them.
__device__ __forceinline__ void combine_block(const Args& args, int t, int col, int lane) {
  const int K = args.K, H = args.n_dim;
  const uint16_t* y = static_cast<const uint16_t*>(args.out);
  const int c = col + 4 * lane;
  const bool fq = args.fq_scale != nullptr;
  const float s = fq ? *args.fq_scale : 1.0f;
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  bool any = false;
  constexpr int KB = 4;   // slots whose rows are loaded together
  for (int k0 = 0; k0 < K; k0 += KB) {
    int p[KB];
    float wt[KB];
    uint2 v[KB];
#pragma unroll
    for (int j = 0; j < KB; ++j) {
      const int k = k0 + j;
      p[j] = k < K ? args.inv_map[(size_t)t * K + k] : -1;
      wt[j] = (k < K && args.topk_w) ? args.topk_w[(size_t)t * K + k] : 1.0f;
    }
#pragma unroll
    for (int j = 0; j < KB; ++j)
      if (p[j] >= 0) v[j] = __ldcg(reinterpret_cast<const uint2*>(y + (size_t)p[j] * H + c));
#pragma unroll
    for (int j = 0; j < KB; ++j) {
      if (p[j] < 0) continue;
      any = true;
      const uint32_t u[2] = {v[j].x, v[j].y};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float yv = __uint_as_float((i & 1) ? (u[i >> 1] & 0xffff0000u) : (u[i >> 1] << 16));
        float r = __fmul_rn(yv, wt[j]);
        if (fq) r = __fdiv_rn(e4m3_to_f32(f32_to_e4m3(__fmul_rn(r, s))), s);
        acc[i] = __fadd_rn(acc[i], r);
      }
    }
  }
  if (any && args.shared_map) {
    const int sp = args.shared_map[t];
    if (sp >= 0) {
      const uint2 sv = __ldcg(reinterpret_cast<const uint2*>(y + (size_t)sp * H + c));
      const uint32_t u[2] = {sv.x, sv.y};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        acc[i] = __fadd_rn(acc[i], __uint_as_float((i & 1) ? (u[i >> 1] & 0xffff0000u) : (u[i >> 1] << 16)));
    }
  }
  uint2 o;
  o.x = (uint32_t)f32_to_bf16(acc[0]) | ((uint32_t)f32_to_bf16(acc[1]) << 16);
  o.y = (uint32_t)f32_to_bf16(acc[2]) | ((uint32_t)f32_to_bf16(acc[3]) << 16);
  *reinterpret_cast<uint2*>(args.comb_out + (size_t)t * H + c) = o;
}

// Tokens with no row anywhere (no valid slot and no shared row) get +0, the combine's value
// for them; warps [w0, w0 + nw) of the grid share the tokens.
__device__ __forceinline__ void zero_rowless_tokens(const Args& args, int w0, int nw, int lane) {
  const int nv = args.n_dim / 8;
  for (int t = w0; t < args.T; t += nw) {
    bool any = false;
    for (int k = lane; k < args.K; k += 32) any |= args.inv_map[(size_t)t * args.K + k] >= 0;
    const bool has_row = __any_sync(0xffffffffu, any) || (args.shared_map && args.shared_map[t] >= 0);
    if (has_row) continue;
    uint4* o = reinterpret_cast<uint4*>(args.comb_out + (size_t)t * args.n_dim);
    for (int v = lane; v < nv; v += 32) o[v] = make_uint4(0, 0, 0, 0);
  }
}

// ------------------------------------------------------------------------ kernel
template <bool FP8, bool SWIGLU, bool FUSE>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmBx, const __grid_constant__ CUtensorMap tmAt,
                        const Args args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr bool M2 = !FP8 && !FUSE;   // two M-tiles per MMA-pipeline unit
  uint8_t* cmn = smem + args.common_off;
  uint64_t* bars = reinterpret_cast<uint64_t*>(cmn);
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + YSTAGES + s); };
  auto bar_tfull = [&](int b) { return smem_u32(bars + 2 * YSTAGES + b); };
  auto bar_tempty = [&](int b) { return smem_u32(bars + 2 * YSTAGES + 2 + b); };
  const uint32_t bar_drain = smem_u32(bars + 2 * YSTAGES + 4);
  const uint32_t bar_drain1 = smem_u32(bars + 2 * YSTAGES + 5);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cmn + SmemLayout::tmem_slot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(cmn + SmemLayout::abort_flag);
  float* costs = reinterpret_cast<float*>(cmn + SmemLayout::costs);
  float* xch = reinterpret_cast<float*>(smem + SmemLayout::xch);
  const int nseg = args.nseg;
  int* cu_s = reinterpret_cast<int*>(cmn + SmemLayout::arrays);
  int* prefix = cu_s + (nseg + 1);
  int* prefix_y = prefix + (nseg + 1);
  uint8_t* stage_out = smem + SmemLayout::stage_out;

  const int mtok = args.max_tokens;
  if (mtok > 0) {
    for (int i = tid; i < nseg; i += THREADS) cu_s[i] = i * mtok + min(max(args.cu[i], 0), mtok);
  } else {
    for (int i = tid; i <= nseg; i += THREADS) cu_s[i] = args.cu[i];
  }
  __syncthreads();
  const int n_tiles = SWIGLU ? (args.n_dim / 2) / 128 : (args.n_dim + BN - 1) / BN;
  // per-segment counts -> exclusive prefixes (warp 0): M-tiles on the MMA pipeline, and
  // streamed segments; plus the modelled time of each kind of work
  if (warp == 0) {
    const int chunk = (nseg + 31) / 32;
    const int s0 = min(nseg, lane * chunk), s1 = min(nseg, s0 + chunk);
    auto len = [&](int s) { return max(0, seg_end(cu_s, s, mtok) - seg_begin(cu_s, s, mtok)); };
    // streaming pays only when every CTA has many units to spread (a static split of a
    // handful of units per CTA is too coarse): at least 16 per CTA, from the M-tile count
    bool stream_on = !FP8 && !FUSE && args.stream;
    if (stream_on) {
      int tiles = 0;
      for (int s = s0; s < s1; ++s) tiles += (len(s) + BM - 1) / BM;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tiles += __shfl_xor_sync(0xffffffffu, tiles, off);
      stream_on = static_cast<long long>(tiles) * n_tiles >= 16ll * gridDim.x;
    }
    auto streamed = [&](int l) { return stream_on && l > 0 && l <= NS; };
    int local = 0, local_y = 0;
    float cx = 0.0f, cy = 0.0f;
    for (int s = s0; s < s1; ++s) {
      const int l = len(s);
      if (streamed(l)) {
        ++local_y;
        cy += COST_STREAM;
      } else {
        const int m = (l + BM - 1) / BM;
        local += M2 ? (m + 1) / 2 : m;
        cx += m == 1 ? COST_SINGLE
                     : (M2 ? COST_MMA2 * static_cast<float>(m / 2) + static_cast<float>(m & 1) * COST_MMA
                           : COST_MMA * static_cast<float>(m));
      }
    }
    int incl = local, incl_y = local_y;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      const int vy = __shfl_up_sync(0xffffffffu, incl_y, off);
      if (lane >= off) {
        incl += v;
        incl_y += vy;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      cx += __shfl_xor_sync(0xffffffffu, cx, off);
      cy += __shfl_xor_sync(0xffffffffu, cy, off);
    }
    int run = incl - local, run_y = incl_y - local_y;
    for (int s = s0; s < s1; ++s) {
      prefix[s] = run;
      prefix_y[s] = run_y;
      const int l = len(s);
      if (streamed(l))
        ++run_y;
      else
        run += M2 ? ((l + BM - 1) / BM + 1) / 2 : (l + BM - 1) / BM;
    }
    if (lane == 31) {
      prefix[nseg] = incl;
      prefix_y[nseg] = incl_y;
    }
    if (lane == 0) {
      costs[0] = cx;
      costs[1] = cy;
    }
  }
  __syncthreads();
  const int total_units = prefix[nseg] * n_tiles;
  const int total_y = prefix_y[nseg] * n_tiles;
  // MMA-pipeline unit u -> segment, N-tile, first row (two-tile units: the prefix counts
  // pairs of M-tiles, so the decoder's row0 is the segment start + (pair index) * BM)
  auto mma_unit = [&](int u) {
    Unit w = decode_unit(u, n_tiles, cu_s, prefix, nseg, mtok,
                         SWIGLU && !FP8 ? (M2 ? MGROUP_GATE_UP_M2 : MGROUP_GATE_UP) : (M2 ? MGROUP_DOWN_M2 : 0));
    if (M2) {
      const int b0 = seg_begin(cu_s, w.seg, mtok);
      w.row0 = b0 + 2 * (w.row0 - b0);
    }
    return w;
  };
  // CTAs [gx, gridDim.x) stream; every CTA derives the same split from the same counts.
  // The estimate ny = the streaming share of the modelled time, then the split near it whose
  // slower role, counted in whole rounds of units (ceil(units / CTAs) x the role's mean unit
  // cost), ends first: a gate/up unit of two M-tiles runs for tens of microseconds, so one
  // more round of units on the MMA pipeline costs more than the proportional model sees.
  int ny = 0;
  if (total_y > 0) {
    const int G = gridDim.x;
    if (total_units == 0) {
      ny = G;
    } else {
      const float f = costs[1] / (costs[0] + costs[1]);
      const int est = min(max(static_cast<int>(f * static_cast<float>(G) + 0.5f), 1), G - 1);
      const float cx_unit = costs[0] / static_cast<float>(prefix[nseg]);
      const float cy_unit = costs[1] / static_cast<float>(prefix_y[nseg]);
      float best = 0.0f;
      for (int c = max(1, est - 8); c <= min(G - 1, est + 8); ++c) {
        const float tx = static_cast<float>((total_units + G - c - 1) / (G - c)) * cx_unit;
        const float ty = static_cast<float>((total_y + c - 1) / c) * cy_unit;
        const float t = fmaxf(tx, ty);
        if (ny == 0 || t < best) {
          best = t;
          ny = c;
        }
      }
    }
  }
  const int gx = static_cast<int>(gridDim.x) - ny;
  const bool y_role = static_cast<int>(blockIdx.x) >= gx;
  // MMA-pipeline CTAs actually used: the fewest that keep the largest per-CTA unit count,
  // so the last round of units is full instead of a few CTAs finishing alone
  // (weight-streaming launches such as decode, where those few cannot draw the HBM
  // bandwidth that all of them share); compute-bound launches keep their critical path.
  int gxu = gx;
  if (total_units > 0 && gx > 0) {
    const int per = (total_units + gx - 1) / gx;
    gxu = min(gx, (total_units + per - 1) / per);
  }
  if (tid == 64) {
    const int nst = y_role ? YSTAGES : (M2 ? STAGES_M2 : STAGES);
    for (int s = 0; s < nst; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull(b), y_role ? y_lanes<SWIGLU>() : 1);   // streaming: one arrival per lane
      mbar_init(bar_tempty(b), y_role ? Y_EPI_WARPS : EPI_WARPS);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_drain1, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  if (FUSE && total_units == 0) {
    // no rows at all: every token's output is +0
    zero_rowless_tokens(args, blockIdx.x * (THREADS / 32) + warp, gridDim.x * (THREADS / 32), lane);
    return;
  }
  // no work: nothing allocated yet
  if (y_role ? static_cast<int>(blockIdx.x) - gx >= total_y
             : static_cast<int>(blockIdx.x) >= min(total_units, gxu))
    return;

  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  constexpr int KE = FP8 ? 128 : 64;  // K elements per stage
  const int kblocks = args.k_dim / KE;
  // Box of 128 weight rows from r0 (a multiple of 128) and K block kb: at (kb * KE, r0) in
  // the row-major weights, or in the tile layout ([tiles * 128, KE], tile (r0 / 128, kb) of
  // a matrix at rows 128 * ((r0 / 128) * kblocks + kb)), where the box is 16 contiguous KB.
  const bool w_tiled = args.w_tiled != 0;
  auto wx = [&](int kb) { return w_tiled ? 0 : kb * KE; };
  auto wy = [&](int r0, int kb) { return w_tiled ? ((r0 >> 7) * kblocks + kb) << 7 : r0; };

  if (y_role) {
    if constexpr (!FP8 && !FUSE) {
      // ================================================ streaming CTA: segments of <= NS rows
      // Unit v: the t-th streamed segment (t = v / n_tiles) and N-tile nt = v % n_tiles.  The
      // two 128-row halves of the weight tile are the A operands of two MMAs (M = 128) that
      // share the segment's NS token rows as B (N = NS).
      // The K blocks of this CTA's units, numbered g = 0, 1, ... in order, run on kLanes
      // lanes of the pipeline (y_lanes, two): lane p (producer thread p, MMA thread p) takes
      // the K blocks with g % kLanes == p, which with two lanes live in the stages of parity
      // p (stage g % YSTAGES, YSTAGES even), and
      // accumulates into its own TMEM columns; the epilogue adds lane 0's sum (even K
      // blocks) and lane 1's (odd K blocks), in that order.  k_dim is a multiple of 128, so
      // a unit has an even number of 64-wide K blocks and g % 2 == kb % 2.  A single MMA
      // thread waits on a barrier between every two groups of eight short MMAs and the
      // tensor pipe idles in those waits; two keep it busy.  TMEM buffer b, lane p: half 0's
      // products in columns [4 NS b + 2 NS p, +NS), half 1's in the next NS columns.
      const int yi = static_cast<int>(blockIdx.x) - gx;
      auto y_unit = [&](int v, int& seg, int& nt) {
        const int t = v / n_tiles;
        nt = v - t * n_tiles;
        int lo = 0, hi = nseg - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (prefix_y[mid] <= t)
            lo = mid;
          else
            hi = mid - 1;
        }
        seg = lo;
      };
      constexpr int kLanes = y_lanes<SWIGLU>();
      if (warp == 0 || (kLanes == 2 && warp == Y_PRODUCER1)) {
        const uint32_t p = warp == 0 ? 0u : 1u;
        if (lane == 0) {
          asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmAt)) : "memory");
          asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
          int stage = 0;
          uint32_t phase = 0, armed = 0, last_parity = 0, g = 0;
          bool ok = true;
          uint64_t wpol;
          asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(wpol));
          for (int v = yi; ok && v < total_y; v += ny) {
            int seg, nt;
            y_unit(v, seg, nt);
            const int row0 = seg_begin(cu_s, seg, mtok);
            const bool extra = seg >= args.num_w;
            const CUtensorMap* mb = extra ? &tmBx : &tmB;
            const int wbase = extra ? 0 : seg * args.n_dim;
            const int rA = SWIGLU ? wbase + nt * 128 : wbase + nt * BN;
            const int rB = SWIGLU ? wbase + args.n_dim / 2 + nt * 128 : rA + 128;
            for (int kb = 0; kb < kblocks; ++kb, ++g) {
              if (g % static_cast<uint32_t>(kLanes) == p) {
                if (!mbar_wait(bar_empty(stage), phase ^ 1, abort_flag, args.dev_status, args.timeout_ns)) {
                  ok = false;
                  break;
                }
                mbar_expect_tx(bar_full(stage), YSTAGE_BYTES);
                armed |= 1u << stage;
                last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                const uint32_t sw = sbase + stage * YSTAGE_BYTES;
                if (STREAM_EVICT_FIRST) {
                  tma_load_2d_hint(sw, mb, wx(kb), wy(rA, kb), bar_full(stage), wpol);
                  tma_load_2d_hint(sw + B_HALF, mb, wx(kb), wy(rB, kb), bar_full(stage), wpol);
                } else {
                  tma_load_2d(sw, mb, wx(kb), wy(rA, kb), bar_full(stage));
                  tma_load_2d(sw + B_HALF, mb, wx(kb), wy(rB, kb), bar_full(stage));
                }
                tma_load_2d(sw + B_BYTES, &tmAt, kb * KE, row0, bar_full(stage));
              }
              if (++stage == YSTAGES) {
                stage = 0;
                phase ^= 1;
              }
            }
          }
          if (!ok) {
            for (int s = 0; s < YSTAGES; ++s)
              if (armed & (1u << s)) mbar_drain(bar_full(s), (last_parity >> s) & 1u);
          }
        }
      } else if (warp == 1 || (kLanes == 2 && warp == Y_ISSUER1)) {
        const uint32_t p = warp == 1 ? 0u : 1u;
        if (lane == 0) {
          constexpr uint32_t idesc = instr_desc_stream();
          const uint32_t drain = p == 0 ? bar_drain : bar_drain1;
          int stage = 0, buf = 0;
          uint32_t phase = 0, tphase = 0, g = 0;
          bool ok = true;
          for (int v = yi; ok && v < total_y; v += ny) {
            if (!mbar_wait(bar_tempty(buf), tphase ^ 1, abort_flag, args.dev_status, args.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t dt = tmem_base + buf * (4 * NS) + p * (2 * NS);
            bool first = true;
            for (int kb = 0; kb < kblocks; ++kb, ++g) {
              if (g % static_cast<uint32_t>(kLanes) == p) {
                if (!mbar_wait(bar_full(stage), phase, abort_flag, args.dev_status, args.timeout_ns)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                const uint32_t sw = sbase + stage * YSTAGE_BYTES;
                const uint32_t st = sw + B_BYTES;
#pragma unroll
                for (int k = 0; k < KB_BYTES / 32; ++k) {
                  const uint32_t acc = !first || k != 0;
                  tc_mma<false>(dt, smem_desc(sw + 32 * k), smem_desc(st + 32 * k), idesc, acc);
                  tc_mma<false>(dt + NS, smem_desc(sw + B_HALF + 32 * k), smem_desc(st + 32 * k), idesc, acc);
                }
                tc_commit(bar_empty(stage));
                first = false;
              }
              if (++stage == YSTAGES) {
                stage = 0;
                phase ^= 1;
              }
            }
            if (!ok) break;
            tc_commit(bar_tfull(buf));  // one of the two arrivals
            if (++buf == 2) {
              buf = 0;
              tphase ^= 1;
            }
          }
          if (!ok) {
            tc_commit(drain);
            mbar_drain(drain, 0);
          }
        }
      } else if (warp >= 2 && warp < 2 + Y_EPI_WARPS) {
        // epilogue: warp w reads TMEM lanes 32 (w % 4).. = weight rows j of both halves
        const int q = warp & 3;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        const int j = 32 * q + lane;
        const int out_cols = SWIGLU ? args.n_dim / 2 : args.n_dim;
        int buf = 0;
        uint32_t tphase = 0;
        for (int v = yi; v < total_y; v += ny) {
          int seg, nt;
          y_unit(v, seg, nt);
          const int row0 = seg_begin(cu_s, seg, mtok), row_end = seg_end(cu_s, seg, mtok);
          if (!mbar_wait(bar_tfull(buf), tphase, abort_flag, args.dev_status, args.timeout_ns)) break;
          tc_fence_after();
          const uint32_t tb = tmem_base + lane_addr + buf * (4 * NS);
          uint32_t d0[NS], d1[NS];
          tmem_ld32(tb, d0);
          tmem_ld32(tb + NS, d1);
          tmem_wait_ld();
          if (kLanes == 2) {
            uint32_t e[NS];
            tmem_ld32(tb + 2 * NS, e);
            tmem_wait_ld();
#pragma unroll
            for (int n = 0; n < NS; ++n) d0[n] = __float_as_uint(__fadd_rn(__uint_as_float(d0[n]), __uint_as_float(e[n])));
            tmem_ld32(tb + 3 * NS, e);
            tmem_wait_ld();
#pragma unroll
            for (int n = 0; n < NS; ++n) d1[n] = __float_as_uint(__fadd_rn(__uint_as_float(d1[n]), __uint_as_float(e[n])));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tempty(buf));
          if (++buf == 2) {
            buf = 0;
            tphase ^= 1;
          }
          const int rows = min(row_end - row0, NS);
          if (SWIGLU) {
            // gate row j in half 0, up row j in half 1: h[token, nt * 128 + j]
            uint16_t* dst = static_cast<uint16_t*>(args.out) + (size_t)row0 * out_cols + nt * 128 + j;
#pragma unroll
            for (int n = 0; n < NS; ++n)
              if (n < rows)
                dst[(size_t)n * out_cols] = f32_to_bf16(silu(__uint_as_float(d0[n])) * __uint_as_float(d1[n]));
          } else {
            const int col = nt * BN + j;
            uint16_t* dst = static_cast<uint16_t*>(args.out) + (size_t)row0 * out_cols + col;
#pragma unroll
            for (int n = 0; n < NS; ++n) {
              if (n < rows) {
                const float rs = args.row_scale ? args.row_scale[row0 + n] : 1.0f;
                float v0 = __uint_as_float(d0[n]), v1 = __uint_as_float(d1[n]);
                if (args.row_scale) {
                  v0 = __fmul_rn(v0, rs);
                  v1 = __fmul_rn(v1, rs);
                }
                if (col < out_cols) dst[(size_t)n * out_cols] = f32_to_bf16(v0);
                if (col + 128 < out_cols) dst[(size_t)n * out_cols + 128] = f32_to_bf16(v1);
              }
            }
          }
        }
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;  // bit s: stage s has been armed at least once
      uint32_t last_parity = 0;  // bit s: parity of the last phase armed on stage s
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gxu) {
        const Unit w = mma_unit(u);
        const bool extra = w.seg >= args.num_w;
        const CUtensorMap* mb = extra ? &tmBx : &tmB;
        const int wbase = extra ? 0 : w.seg * args.n_dim;
        const int rA = SWIGLU ? wbase + w.nt * 128 : wbase + w.nt * BN;
        const int rB = SWIGLU ? wbase + args.n_dim / 2 + w.nt * 128 : rA + 128;
        // two-tile units: the second M-tile's rows when the segment has them
        const bool two = M2 && w.row0 + BM < w.row_end;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(bar_empty(stage), phase ^ 1, abort_flag, args.dev_status, args.timeout_ns)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar_full(stage), M2 ? (two ? STAGE_M2_BYTES : STAGE_M2_BYTES - A_BYTES) : STAGE_TX);
          armed |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (M2) {
            // stage: [A rows of M-tile 0 | A rows of M-tile 1 | 256 weight rows]
            const uint32_t sa = sbase + stage * STAGE_M2_BYTES;
            const uint32_t sb = sa + 2 * A_BYTES;
            tma_load_2d(sa, &tmA, kb * KE, w.row0, bar_full(stage));
            if (two) tma_load_2d(sa + A_BYTES, &tmA, kb * KE, w.row0 + BM, bar_full(stage));
            tma_load_2d(sb, mb, wx(kb), wy(rA, kb), bar_full(stage));
            tma_load_2d(sb + B_HALF, mb, wx(kb), wy(rB, kb), bar_full(stage));
          } else {
            const uint32_t sa = sbase + SmemLayout::a + stage * A_BYTES;
            const uint32_t sb = sbase + SmemLayout::b + stage * B_BYTES;
            tma_load_2d(sa, &tmA, kb * KE, w.row0, bar_full(stage));
            tma_load_2d(sb, mb, wx(kb), wy(rA, kb), bar_full(stage));
            tma_load_2d(sb + B_HALF, mb, wx(kb), wy(rB, kb), bar_full(stage));
          }
          if (++stage == (M2 ? STAGES_M2 : STAGES)) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // wait for the copies this CTA still has in flight before its shared memory goes away
        for (int s = 0; s < (M2 ? STAGES_M2 : STAGES); ++s)
          if (armed & (1u << s)) mbar_drain(bar_full(s), (last_parity >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc<FP8>();
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t tphase = 0;
      bool ok = true;
      if constexpr (M2) {
        // two-tile units: accumulator t (TMEM columns [BN t, +BN)) holds M-tile t, one buffer.
        // At a unit's first K step the MMAs into accumulator 0 wait for the epilogue to have
        // read it, those into accumulator 1 for the second read, so the epilogue's work on
        // M-tile 0 overlaps the new unit's first MMAs.
        for (int u = blockIdx.x; ok && u < total_units; u += gxu) {
          const Unit w = mma_unit(u);
          const bool two = w.row0 + BM < w.row_end;
          for (int kb = 0; kb < kblocks; ++kb) {
            if (kb == 0) {
              if (!mbar_wait(bar_tempty(0), tphase ^ 1, abort_flag, args.dev_status, args.timeout_ns)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            if (!mbar_wait(bar_full(stage), phase, abort_flag, args.dev_status, args.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = sbase + stage * STAGE_M2_BYTES;
            const uint32_t sb = sa + 2 * A_BYTES;
#pragma unroll
            for (int k = 0; k < KB_BYTES / 32; ++k)
              tc_mma<false>(tmem_base, smem_desc(sa + 32 * k), smem_desc(sb + 32 * k), idesc, (kb | k) != 0);
            if (kb == 0) {
              if (!mbar_wait(bar_tempty(1), tphase ^ 1, abort_flag, args.dev_status, args.timeout_ns)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            if (two) {
#pragma unroll
              for (int k = 0; k < KB_BYTES / 32; ++k)
                tc_mma<false>(tmem_base + BN, smem_desc(sa + A_BYTES + 32 * k), smem_desc(sb + 32 * k), idesc,
                              (kb | k) != 0);
            }
            tc_commit(bar_empty(stage));
            if (++stage == STAGES_M2) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          tc_commit(bar_tfull(0));
          tphase ^= 1;
        }
      } else {
        for (int u = blockIdx.x; ok && u < total_units; u += gxu) {
          for (int kb = 0; kb < kblocks; ++kb) {
            const bool round_start = FP8 || kb == 0;
            if (round_start) {
              if (!mbar_wait(bar_tempty(buf), tphase ^ 1, abort_flag, args.dev_status, args.timeout_ns)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            if (!mbar_wait(bar_full(stage), phase, abort_flag, args.dev_status, args.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = sbase + SmemLayout::a + stage * A_BYTES;
            const uint32_t sb = sbase + SmemLayout::b + stage * B_BYTES;
            const uint32_t dt = tmem_base + buf * BN;
#pragma unroll
            for (int k = 0; k < KB_BYTES / 32; ++k) {
              const uint32_t acc = (FP8 ? k : (kb | k)) != 0;
              tc_mma<FP8>(dt, smem_desc(sa + 32 * k), smem_desc(sb + 32 * k), idesc, acc);
            }
            tc_commit(bar_empty(stage));
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
            const bool round_end = FP8 || kb == kblocks - 1;
            if (round_end) {
              tc_commit(bar_tfull(buf));
              if (++buf == 2) {
                buf = 0;
                tphase ^= 1;
              }
            }
          }
        }
      }
      if (!ok) {
        tc_commit(bar_drain);  // arrives once every MMA issued so far has completed
        mbar_drain(bar_drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;               // TMEM subpartition this warp may access
    const int half = (warp - 2) >> 2;     // which half of the tile's columns
    const int r_in_tile = 32 * q + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    const int kbs_total = kblocks;
    int buf = 0;
    uint32_t tphase = 0;
    const int out_cols = SWIGLU ? args.n_dim / 2 : args.n_dim;
    if (FUSE) {
      // while the first accumulator fills: +0 rows for the tokens no unit will touch
      const int active = min(gxu, total_units);
      zero_rowless_tokens(args, blockIdx.x * EPI_WARPS + (warp - 2), active * EPI_WARPS, lane);
    }
    if constexpr (M2) {
      // two-tile units (BF16, not fused): read accumulator 0, free it, compute and store
      // M-tile 0's rows; then accumulator 1 (freed at once when the unit has one M-tile) and
      // M-tile 1
      for (int u = blockIdx.x; u < total_units; u += gxu) {
        const Unit w = mma_unit(u);
        const bool two = w.row0 + BM < w.row_end;
        const int col0 = SWIGLU ? w.nt * 128 + 64 * half : w.nt * BN + 128 * half;
        const bool cols_ok = col0 < out_cols;
        if (!mbar_wait(bar_tfull(0), tphase, abort_flag, args.dev_status, args.timeout_ns)) break;
        tc_fence_after();
        for (int t = 0; t < 2; ++t) {
          if (t == 1 && !two) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_tempty(1));
            break;
          }
          float acc[128];
          const uint32_t tb = tmem_base + lane_addr + t * BN;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int tcol = SWIGLU ? (c < 2 ? 64 * half + 32 * c : 128 + 64 * half + 32 * (c - 2))
                                    : 128 * half + 32 * c;
            uint32_t r[32];
            tmem_ld32(tb + tcol, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[32 * c + i] = __uint_as_float(r[i]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tempty(t));
          const int trow0 = w.row0 + t * BM;   // first row of M-tile t
          const int row = trow0 + r_in_tile;
          if (SWIGLU) {
            if (row < w.row_end && cols_ok) {
              float h[64];
#pragma unroll
              for (int i = 0; i < 64; ++i) h[i] = silu(acc[i]) * acc[64 + i];
              store_h_bf16(h, static_cast<uint16_t*>(args.out) + (size_t)row * out_cols + col0);
            }
          } else if (cols_ok) {
            if (args.row_scale) {
              // router weight of each permuted row, applied to the float32 accumulator
              const float rs = row < w.row_end ? args.row_scale[row] : 0.0f;
#pragma unroll
              for (int i = 0; i < 128; ++i) acc[i] = __fmul_rn(acc[i], rs);
            }
            const int rows_here = w.row_end - (trow0 + 32 * q);   // rows of this warp's 32 in the segment
            store_rows_bf16(acc, stage_out + (warp - 2) * STAGE_OUT_BYTES, lane, rows_here,
                            static_cast<uint16_t*>(args.out), trow0 + 32 * q, out_cols, col0);
          }
        }
        tphase ^= 1;
      }
    } else {
      for (int u = blockIdx.x; u < total_units; u += gxu) {
        const Unit w = mma_unit(u);
        const int row = w.row0 + r_in_tile;
        const bool row_ok = row < w.row_end;
        // first output column this thread covers and whether that 128-column block exists
        const int col0 = SWIGLU ? w.nt * 128 + 64 * half : w.nt * BN + 128 * half;
        const bool cols_ok = col0 < out_cols;
        float acc[128];
        if (FP8) {
#pragma unroll
          for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
        }
        const bool extra = w.seg >= args.num_w;
        // FP8: a warp whose 32 rows all lie past the segment's end has nothing to promote in
        // any of the K rounds and only keeps the TMEM hand-off going (decode segments often
        // hold a few rows).  BF16 has one round per tile and keeps the plain path.
        const bool warp_live = !FP8 || w.row0 + 32 * q < w.row_end;
        int rounds = FP8 ? kbs_total : 1;
        bool ok = true;
        // FP8 weight scales of this unit: one row of K-block scales for each 128 weight rows
        const float* wsc = nullptr;
        size_t ws0 = 0, ws1 = 0;
        if (FP8) {
          wsc = extra ? args.wx_scales : args.w_scales + (size_t)w.seg * (args.n_dim / 128) * kbs_total;
          if (SWIGLU) {
            ws0 = (size_t)w.nt * kbs_total;                            // gate rows
            ws1 = (size_t)(args.n_dim / 256 + w.nt) * kbs_total;       // up rows
          } else {
            ws0 = ws1 = (size_t)((w.nt * BN + 128 * half) / 128) * kbs_total;
          }
        }
        for (int rd = 0; rd < rounds; ++rd) {
          if (!mbar_wait(bar_tfull(buf), tphase, abort_flag, args.dev_status, args.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tb = tmem_base + lane_addr + buf * BN;
          if (!warp_live) {
            // nothing to read
          } else if (FP8) {
            // promotion of this K block: acc += partial * (s_a[row, kb] * s_w[block, kb])
            const float sa = row_ok ? args.a_scales[(size_t)row * kbs_total + rd] : 0.0f;
            const float s0 = cols_ok ? wsc[ws0 + rd] * sa : 0.0f;
            const float s1 = cols_ok ? wsc[ws1 + rd] * sa : 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int tcol = SWIGLU ? (c < 2 ? 64 * half + 32 * c : 128 + 64 * half + 32 * (c - 2))
                                      : 128 * half + 32 * c;
              uint32_t r[32];
              tmem_ld32(tb + tcol, r);
              tmem_wait_ld();
              const float sc = (SWIGLU && c >= 2) ? s1 : s0;
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[32 * c + i] = fmaf(__uint_as_float(r[i]), sc, acc[32 * c + i]);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int tcol = SWIGLU ? (c < 2 ? 64 * half + 32 * c : 128 + 64 * half + 32 * (c - 2))
                                      : 128 * half + 32 * c;
              uint32_t r[32];
              tmem_ld32(tb + tcol, r);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[32 * c + i] = __uint_as_float(r[i]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tempty(buf));
          if (++buf == 2) {
            buf = 0;
            tphase ^= 1;
          }
        }
        // FP8 SwiGLU: the eight warps exchange row maxima through a named barrier below, so
        // they agree on leaving (one reduction per unit on every warp) before any of them does
        if (FP8 && SWIGLU) {
          if (bar_red_or(1, 32 * EPI_WARPS, !ok)) break;
        } else if (!ok) {
          break;
        }
        // ---- tile epilogue from registers
        if (SWIGLU) {
          float h[64];
#pragma unroll
          for (int i = 0; i < 64; ++i) h[i] = silu(acc[i]) * acc[64 + i];
          if (!FP8) {
            if (row_ok && cols_ok) store_h_bf16(h, static_cast<uint16_t*>(args.out) + (size_t)row * out_cols + col0);
          } else {
            // 1x128 block of h = this thread's 64 columns + the partner half's 64
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(h[i]));
            xch[half * 128 + r_in_tile] = amax;
            asm volatile("bar.sync 1, 256;" ::: "memory");
            amax = fmaxf(amax, xch[(1 - half) * 128 + r_in_tile]);
            asm volatile("bar.sync 1, 256;" ::: "memory");
            const float s = block_scale(amax);
            if (row_ok && cols_ok) {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(args.out) + (size_t)row * out_cols + col0);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  uint32_t word = 0;
#pragma unroll
                  for (int b = 0; b < 4; ++b) word |= (uint32_t)f32_to_e4m3(__fdiv_rn(h[16 * v + 4 * j + b], s)) << (8 * b);
                  o[j] = word;
                }
                dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
              }
              if (half == 0) args.out_scales[(size_t)row * (out_cols / 128) + w.nt] = s;
            }
          }
        } else if (cols_ok) {
          if (args.row_scale) {
            // router weight of each permuted row, applied to the float32 accumulator
            const float rs = row_ok ? args.row_scale[row] : 0.0f;
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = __fmul_rn(acc[i], rs);
          }
          const int rows_here = w.row_end - (w.row0 + 32 * q);   // rows of this warp's 32 in the segment
          store_rows_bf16(acc, stage_out + (warp - 2) * STAGE_OUT_BYTES, lane, rows_here,
                          static_cast<uint16_t*>(args.out), w.row0 + 32 * q, out_cols, col0);
          if (FUSE) {
            // Rows [row0 + 32q, + rows_here) x columns [col0, col0 + 128) are stored.  Each lane
            // counts its row in the (token, 128-column block) counter; the lane whose count
            // completes the token's rows (its valid slots + its shared row) has its warp sum
            // the block.  Every lane's stores are fenced before the counts (release); the
            // summing warp fences again before it reads the rows (acquire).  No CTA waits.
            __threadfence();
            __syncwarp();
            int done_t = -1;
            if (lane < rows_here) {
              const int src = args.src_row[w.row0 + 32 * q + lane];
              const int TK = args.T * args.K;
              const int t = src < TK ? src / args.K : src - TK;
              if (src >= 0 && t < args.T) {
                // rows of token t: its valid slots and its shared row (loads issued together)
                int target = 0;
                for (int k0 = 0; k0 < args.K; k0 += 8) {
                  int pv[8];
#pragma unroll
                  for (int j = 0; j < 8; ++j) pv[j] = k0 + j < args.K ? args.inv_map[(size_t)t * args.K + k0 + j] : -1;
#pragma unroll
                  for (int j = 0; j < 8; ++j) target += pv[j] >= 0;
                }
                if (args.shared_map && args.shared_map[t] >= 0) ++target;
                int32_t* cnt = args.counters + (size_t)t * (args.n_dim / 128) + col0 / 128;
                if (atomicAdd(cnt, 1) == target - 1) {
                  *cnt = 0;   // every row of this block has arrived: reset for the next call
                  done_t = t;
                }
              }
            }
            unsigned m = __ballot_sync(0xffffffffu, done_t >= 0);
            if (m) __threadfence();
            while (m) {
              const int l = __ffs(m) - 1;
              m &= m - 1;
              combine_block(args, __shfl_sync(0xffffffffu, done_t, l), col0, lane);
            }
          }
        }
      }
    }
  }
  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
}

// ---------------------------------------------------------------------- host side
// cuTensorMapEncodeTiled from the CUDA driver API, looked up once (a function-local static:
// thread-safe initialisation when several host threads make their first call together).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

bool make_map(CUtensorMap* m, const void* ptr, bool fp8, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t esz = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(KB_BYTES / esz), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool FP8, bool SWIGLU, bool FUSE = false>
moe_status_t launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& bx, const CUtensorMap& at,
                    const Args& args, int grid, size_t smem, cudaStream_t s) {
  auto kern = grouped_gemm_kernel<FP8, SWIGLU, FUSE>;
  static std::atomic<unsigned long long> attr_done{0};
  if (!once_per_device(attr_done, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX) == cudaSuccess;
      }))
    return MOE_ERR_CUDA;
  kern<<<grid, THREADS, smem, s>>>(a, b, bx, at, args);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

}  // namespace gg
}  // namespace moe

namespace moe {
namespace gg {
struct FuseIn {
  const int32_t* src_row;
  const int32_t* inv_map;
  const float* topk_w;
  const int32_t* shared_map;
  const float* fq_scale;
  uint16_t* out;
  int32_t* counters;
  int T, K;
};

// max_tokens == 0: segments from cu_seqlens over rows_cap rows; > 0: batched segments
// (bounds = masked_m) over rows_cap = num_segments * max_tokens rows.  fuse: the down
// projection with the combine fused into its epilogue.
static moe_status_t gemm_impl(const void* a, const float* a_scales, const int32_t* cu_seqlens, int max_tokens,
                              int num_segments, int rows_cap, int k_dim, int n_dim, const void* w,
                              const float* w_scales, int num_w, const void* w_extra, const float* w_extra_scales,
                              moe_dtype_t dtype, moe_epilogue_t epilogue, void* out, float* out_scales,
                              int32_t* dev_status, const float* row_scale, void* stream,
                              const FuseIn* fuse = nullptr, unsigned long long timeout_ns = TIMEOUT_NS,
                              bool pairs = false) {
  // MOE_W_TILED in dtype: the weights are in the tile layout of moe_pack_weights
  const bool tiled = (static_cast<int>(dtype) & MOE_W_TILED) != 0;
  dtype = static_cast<moe_dtype_t>(static_cast<int>(dtype) & ~MOE_W_TILED);
  const bool fp8 = dtype == MOE_E4M3;
  const bool swiglu = epilogue == MOE_EPI_SWIGLU;
  if (dtype != MOE_BF16 && dtype != MOE_E4M3) return MOE_ERR_ARG;
  if (epilogue != MOE_EPI_NONE && epilogue != MOE_EPI_SWIGLU) return MOE_ERR_ARG;
  if (num_segments < 0 || num_segments > MAX_SEG || rows_cap < 0 || num_w < 0) return MOE_ERR_ARG;
  if (num_segments > num_w + (w_extra ? 1 : 0)) return MOE_ERR_ARG;
  if (k_dim <= 0 || k_dim % 128 != 0 || n_dim <= 0 || n_dim % 128 != 0) return MOE_ERR_ARG;
  if (swiglu && (n_dim % 256 != 0)) return MOE_ERR_ARG;
  if (swiglu && row_scale) return MOE_ERR_ARG;
  if (fuse) {
    if (swiglu || fuse->T < 0 || fuse->K < 1 || fuse->K > kMaxTopK) return MOE_ERR_ARG;
    if (fuse->T == 0) return MOE_OK;
    if (!fuse->src_row || !fuse->inv_map || !fuse->out || !fuse->counters) return MOE_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(fuse->out) & 15) return MOE_ERR_ARG;
    // every token's output is written by this call, so it needs at least one row of capacity
    if (num_segments == 0 || rows_cap == 0) return MOE_ERR_ARG;
    if ((long long)fuse->T * fuse->K + fuse->T > 0x7fffffffll) return MOE_ERR_ARG;
  }
  if (num_segments == 0 || rows_cap == 0) return MOE_OK;
  if (!a || !cu_seqlens || !out || (num_w > 0 && !w)) return MOE_ERR_ARG;
  if (fp8 && (!a_scales || (num_w > 0 && !w_scales) || (w_extra && !w_extra_scales))) return MOE_ERR_ARG;
  if (fp8 && swiglu && !out_scales) return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(w_extra) |
       reinterpret_cast<uintptr_t>(out)) & 15)
    return MOE_ERR_ARG;
  if ((uint64_t)num_w * n_dim > 0x7fffffffull) return MOE_ERR_ARG;
  // tile layout: box row coordinates up to num_w * n_dim * k_dim / KE stay in int
  const uint64_t ke_el = fp8 ? 128 : 64;
  if (tiled && (pairs || (uint64_t)std::max(num_w, 1) * n_dim * (k_dim / ke_el) > 0x7fffffffull))
    return pairs ? MOE_ERR_UNSUPPORTED : MOE_ERR_ARG;
  Args args;
  args.cu = cu_seqlens;
  args.max_tokens = max_tokens;
  args.nseg = num_segments;
  args.rows_cap = rows_cap;
  args.k_dim = k_dim;
  args.n_dim = n_dim;
  args.num_w = num_w;
  args.a_scales = a_scales;
  args.w_scales = w_scales;
  args.wx_scales = w_extra_scales;
  args.out = out;
  args.out_scales = out_scales;
  args.dev_status = dev_status;
  args.row_scale = row_scale;
  args.src_row = fuse ? fuse->src_row : nullptr;
  args.inv_map = fuse ? fuse->inv_map : nullptr;
  args.topk_w = fuse ? fuse->topk_w : nullptr;
  args.shared_map = fuse ? fuse->shared_map : nullptr;
  args.fq_scale = fuse ? fuse->fq_scale : nullptr;
  args.comb_out = fuse ? fuse->out : nullptr;
  args.counters = fuse ? fuse->counters : nullptr;
  args.T = fuse ? fuse->T : 0;
  args.K = fuse ? fuse->K : 1;
  args.timeout_ns = timeout_ns;
  args.w_tiled = tiled ? 1 : 0;
  cudaStream_t s = as_stream(stream);
  // BF16 on CTA pairs with the 2-SM MMA (gemm2sm.cu), when asked for
  if (pairs) {
    if (fp8 || fuse) return MOE_ERR_UNSUPPORTED;
    args.stream = 1;
    args.common_off = 0;
    return launch_2sm(a, rows_cap, k_dim, n_dim, w, num_w, w_extra, swiglu, args, true, s);
  }
  CUtensorMap ma, mb, mbx, mat;
  if (!make_map(&ma, a, fp8, k_dim, rows_cap)) return MOE_ERR_CUDA;
  if (!make_map(&mat, a, fp8, k_dim, rows_cap, NS)) return MOE_ERR_CUDA;
  const void* wb = num_w > 0 ? w : w_extra;
  const uint64_t wrows = num_w > 0 ? (uint64_t)num_w * n_dim : (uint64_t)n_dim;
  // weights: [rows, k_dim] row-major, or the tile layout viewed as [rows * k_dim / KE, KE]
  const uint64_t kt = tiled ? (uint64_t)k_dim / ke_el : 1;
  const uint64_t w_inner = tiled ? ke_el : (uint64_t)k_dim;
  if (!make_map(&mb, wb, fp8, w_inner, wrows * kt)) return MOE_ERR_CUDA;
  if (w_extra) {
    if (!make_map(&mbx, w_extra, fp8, w_inner, (uint64_t)n_dim * kt)) return MOE_ERR_CUDA;
  } else {
    mbx = mb;
  }
  // grid: one CTA per SM, never more than the largest possible number of tiles
  const int n_tiles = swiglu ? (n_dim / 2) / 128 : (n_dim + BN - 1) / BN;
  const long long max_units = ((long long)(rows_cap + BM - 1) / BM + num_segments) * n_tiles;
  const int grid = (int)std::min<long long>(num_sms(), max_units);
  // streaming CTAs for short segments: BF16, not fused, and a grid wide enough to split
  bool stream_on = !fp8 && !fuse && grid >= 16;
  int common_off = stream_on ? std::max(SmemLayout::x_end, SmemLayout::y_end) : SmemLayout::x_end;
  size_t smem = SmemLayout::bytes(common_off, num_segments);
  if (stream_on && smem > (size_t)SMEM_MAX) {
    stream_on = false;
    common_off = SmemLayout::x_end;
    smem = SmemLayout::bytes(common_off, num_segments);
  }
  if (smem > (size_t)SMEM_MAX) return MOE_ERR_ARG;
  args.stream = stream_on ? 1 : 0;
  args.common_off = common_off;
  if (fuse)
    return fp8 ? launch<true, false, true>(ma, mb, mbx, mat, args, grid, smem, s)
               : launch<false, false, true>(ma, mb, mbx, mat, args, grid, smem, s);
  if (fp8)
    return swiglu ? launch<true, true>(ma, mb, mbx, mat, args, grid, smem, s)
                  : launch<true, false>(ma, mb, mbx, mat, args, grid, smem, s);
  return swiglu ? launch<false, true>(ma, mb, mbx, mat, args, grid, smem, s)
                : launch<false, false>(ma, mb, mbx, mat, args, grid, smem, s);
}
}  // namespace gg
}  // namespace moe

// Tile layout (moe_pack_weights): a copy of w [rows, k] (rows % 128 == 0, rows of 128-byte
// tile rows) in which the tile of 128 rows x 128 bytes at (row block rb, K block kb) is
// contiguous, at byte ((rb * kbn + kb) * 128) * 128, kbn = row bytes / 128.  Each thread
// writes 16-byte pieces in destination order (a tile row is 8 of them).
namespace moe {
__global__ void __launch_bounds__(256) pack_tiles_kernel(const uint4* __restrict__ w, uint4* __restrict__ t,
                                                         uint64_t total, uint32_t k16) {
  const uint32_t kbn = k16 / 8;
  for (uint64_t d = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; d < total;
       d += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t j = static_cast<uint32_t>(d & 7);
    const uint32_t rr = static_cast<uint32_t>((d >> 3) & 127);
    const uint64_t tile = d >> 10;
    const uint64_t kb = tile % kbn, rb = tile / kbn;
    t[d] = w[(rb * 128 + rr) * k16 + kb * 8 + j];
  }
}
}  // namespace moe

extern "C" moe_status_t moe_pack_weights(const void* w, int E, int N, int K, moe_dtype_t dtype, void* w_tiled,
                                         void* stream) {
  if (dtype != MOE_BF16 && dtype != MOE_E4M3) return MOE_ERR_ARG;
  if (E < 0 || N < 0 || K < 0 || N % 128 != 0 || K % 128 != 0) return MOE_ERR_ARG;
  const uint64_t esz = dtype == MOE_E4M3 ? 1 : 2;
  const uint64_t bytes = (uint64_t)E * N * K * esz;
  if (bytes == 0) return MOE_OK;
  if (!w || !w_tiled || ((reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(w_tiled)) & 15))
    return MOE_ERR_ARG;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(w), b0 = reinterpret_cast<uintptr_t>(w_tiled);
  if (a0 < b0 + bytes && b0 < a0 + bytes) return MOE_ERR_ARG;   // not in place, no overlap
  const uint64_t total = bytes / 16;
  const int blocks = (int)std::min<uint64_t>((total + 255) / 256, (uint64_t)moe::num_sms() * 8);
  moe::pack_tiles_kernel<<<blocks, 256, 0, moe::as_stream(stream)>>>(
      static_cast<const uint4*>(w), static_cast<uint4*>(w_tiled), total, static_cast<uint32_t>(K * esz / 16));
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

extern "C" moe_status_t moe_grouped_gemm_ex(const void* a, const float* a_scales, const int32_t* cu_seqlens,
                                            int num_segments, int rows_cap, int k_dim, int n_dim, const void* w,
                                            const float* w_scales, int num_w, const void* w_extra,
                                            const float* w_extra_scales, moe_dtype_t dtype, moe_epilogue_t epilogue,
                                            void* out, float* out_scales, int32_t* dev_status,
                                            const float* row_scale, void* stream) {
  return moe::gg::gemm_impl(a, a_scales, cu_seqlens, 0, num_segments, rows_cap, k_dim, n_dim, w, w_scales, num_w,
                            w_extra, w_extra_scales, dtype, epilogue, out, out_scales, dev_status, row_scale, stream);
}

// Test hook, deliberately absent from the public header: moe_grouped_gemm_ex (pairs = 0) or
// moe_grouped_gemm_pairs (pairs = 1) with the limit of each pipeline wait given in
// nanoseconds instead of the built-in 2 s, so that a test can make a wait run out and check
// the abort path (MOE_DEV_PIPELINE_TIMEOUT set, the call returns, the next call is
// unaffected) without faulting or hanging anything.
extern "C" moe_status_t moe_testing_grouped_gemm_wait_limit(
    const void* a, const float* a_scales, const int32_t* cu_seqlens, int num_segments, int rows_cap, int k_dim,
    int n_dim, const void* w, const float* w_scales, int num_w, const void* w_extra, const float* w_extra_scales,
    moe_dtype_t dtype, moe_epilogue_t epilogue, void* out, float* out_scales, int32_t* dev_status,
    const float* row_scale, unsigned long long wait_limit_ns, int pairs, void* stream) {
  return moe::gg::gemm_impl(a, a_scales, cu_seqlens, 0, num_segments, rows_cap, k_dim, n_dim, w, w_scales, num_w,
                            w_extra, w_extra_scales, dtype, epilogue, out, out_scales, dev_status, row_scale, stream,
                            nullptr, wait_limit_ns, pairs != 0);
}

extern "C" moe_status_t moe_grouped_gemm_pairs(const void* a, const int32_t* cu_seqlens, int num_segments,
                                               int rows_cap, int k_dim, int n_dim, const void* w, int num_w,
                                               const void* w_extra, moe_epilogue_t epilogue, void* out,
                                               int32_t* dev_status, const float* row_scale, void* stream) {
  return moe::gg::gemm_impl(a, nullptr, cu_seqlens, 0, num_segments, rows_cap, k_dim, n_dim, w, nullptr, num_w,
                            w_extra, nullptr, MOE_BF16, epilogue, out, nullptr, dev_status, row_scale, stream, nullptr,
                            moe::gg::TIMEOUT_NS, true);
}

extern "C" moe_status_t moe_grouped_gemm_combine(
    const void* a, const float* a_scales, const int32_t* seg, int num_segments, int max_tokens, int rows_cap,
    int k_dim, int n_dim, const void* w, const float* w_scales, int num_w, const void* w_extra,
    const float* w_extra_scales, moe_dtype_t dtype, uint16_t* y, const float* row_scale, const int32_t* src_row,
    const int32_t* inv_map, const float* topk_w, int T, int K, const int32_t* shared_map, const float* fq_scale,
    uint16_t* out, int32_t* counters, int32_t* dev_status, void* stream) {
  if (max_tokens < 0) return MOE_ERR_ARG;
  if (max_tokens > 0) {
    if (num_segments < 0 || (long long)num_segments * max_tokens > 0x7fffffffll) return MOE_ERR_ARG;
    rows_cap = num_segments * max_tokens;
  }
  const moe::gg::FuseIn f{src_row, inv_map, topk_w, shared_map, fq_scale, out, counters, T, K};
  return moe::gg::gemm_impl(a, a_scales, seg, max_tokens, num_segments, rows_cap, k_dim, n_dim, w, w_scales, num_w,
                            w_extra, w_extra_scales, dtype, MOE_EPI_NONE, y, nullptr, dev_status, row_scale, stream,
                            &f);
}

extern "C" moe_status_t moe_grouped_gemm_batched(const void* a, const float* a_scales, const int32_t* masked_m,
                                                 int num_segments, int max_tokens, int k_dim, int n_dim,
                                                 const void* w, const float* w_scales, int num_w,
                                                 const void* w_extra, const float* w_extra_scales, moe_dtype_t dtype,
                                                 moe_epilogue_t epilogue, void* out, float* out_scales,
                                                 int32_t* dev_status, const float* row_scale, void* stream) {
  if (max_tokens < 1 || num_segments < 0 || (long long)num_segments * max_tokens > 0x7fffffffll) return MOE_ERR_ARG;
  return moe::gg::gemm_impl(a, a_scales, masked_m, max_tokens, num_segments, num_segments * max_tokens, k_dim,
                            n_dim, w, w_scales, num_w, w_extra, w_extra_scales, dtype, epilogue, out, out_scales,
                            dev_status, row_scale, stream);
}

extern "C" moe_status_t moe_grouped_gemm(const void* a, const float* a_scales, const int32_t* cu_seqlens,
                                         int num_segments, int rows_cap, int k_dim, int n_dim, const void* w,
                                         const float* w_scales, int num_w, const void* w_extra,
                                         const float* w_extra_scales, moe_dtype_t dtype, moe_epilogue_t epilogue,
                                         void* out, float* out_scales, int32_t* dev_status, void* stream) {
  return moe_grouped_gemm_ex(a, a_scales, cu_seqlens, num_segments, rows_cap, k_dim, n_dim, w, w_scales, num_w,
                             w_extra, w_extra_scales, dtype, epilogue, out, out_scales, dev_status, nullptr, stream);
}
