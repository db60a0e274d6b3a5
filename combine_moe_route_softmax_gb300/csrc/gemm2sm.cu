// BF16 grouped GEMM on CTA pairs with the 2-SM MMA (tcgen05.mma.cta_group::2), behind
// moe_grouped_gemm_pairs.  It computes the same products in the same order as the
// single-CTA kernel (gemm.cu), and its output is identical bit for bit.  Measured on GB300:
// per SM its MMA pipeline ran a K step in 0.36 us against 0.40 us for one-tile units of one
// CTA, but a streamed unit costs its two SMs 1.7 times the SM time of a single streaming
// CTA; since the single-CTA kernel moved to units of two M-tiles it is faster still (layer
// 5.34 against 6.04 ms per step on the prefill expert mix, one box).  The layer uses the
// single-CTA kernel.
//
// MoonEP page: the experts run as grouped matmuls (gate, up, down) over the cu_seqlens
// segments.  This kernel computes them for BF16 operands on pairs of CTAs (clusters of two
// SMs).  One MMA of the pair has M = 256: each CTA holds 128 of the M rows of A in its own
// shared memory and half of the N rows of B, and each CTA's tensor memory receives its own
// 128 rows of the product.  Per 64-wide K step a CTA therefore fills 32 KB of shared memory
// (16 KB of A, 16 KB of B) for 128 x 256 products, where a CTA working alone fills 48 KB
// for the same work; on the prefill mix the single-CTA tile's tensor pipe waits about a
// fifth of its cycles for operand tiles coming from L2, and a third fewer bytes per step
// recovers about a tenth of the time.  No copy is multicast: every CTA loads only its own
// tiles.
//
// Two roles, both on pairs.
//   MMA pipeline (segments of more than NS rows): a unit is two M-tiles of one segment
//     (CTA rank r takes M-tile 2 mp + r) and one N-tile of 256 weight rows (SwiGLU: 128 gate
//     rows on rank 0 and the matching 128 up rows on rank 1, so each CTA's accumulator holds
//     g and u side by side for its rows; plain: weight rows [256 nt + 128 r, +128) on rank r).
//   Streaming pairs (segments of at most NS rows, when the launch has many units): the
//     weights are the M operand (128 rows per CTA) and the segment's rows the N operand
//     (N = NS, NS / 2 rows per CTA), through a 10-stage ring of 18 KB stages per CTA run as
//     two lanes (alternate K blocks, two TMA threads per CTA, two MMA threads in the
//     leader, even and odd K blocks summed apart and then added).  For
//     SwiGLU rank r holds gate rows [128 nt + 64 r, +64) and the matching up rows, so its
//     tensor memory lanes 0-63 hold g and lanes 64-127 u of the same 64 output columns.
//
// Hand-offs inside a pair.  Rank 0 (the leader) issues every MMA.  Both CTAs' TMA copies of
// a stage complete on the leader's full barrier (the CTA-pair form of the copy may signal a
// barrier of either CTA of the pair), which the leader's producer arms with the bytes of
// both.  The leader's tcgen05.commit arrives on both CTAs' empty (stage free) and tfull
// (accumulator ready) barriers; the epilogue warps of both CTAs arrive on the leader's
// tempty barrier (accumulator drained).  A stage thus costs one cross-CTA hop each way.
// (A first version had rank 1's copies complete on its own barrier and one thread pass each
// completion on with a remote arrive: that hop, paid once per stage, held both roles to
// about 0.8-1.1 us per K step.)
//
// Every mbarrier wait is bounded (Args::timeout_ns of globaltimer); on expiry a CTA sets
// MOE_DEV_PIPELINE_TIMEOUT, raises its own and its partner's abort flag and every role leaves
// its loop.  The leader then waits (bounded) for the stages it armed, which covers both
// CTAs' copies of those stages, and for its MMAs; rank 1, whose copies it cannot observe
// itself, waits a grace period of 1 ms (copies of a few tens of KB land within microseconds)
// before both CTAs meet at a cluster barrier and free the tensor memory.
#include "gemm_common.cuh"

namespace moe {
namespace gg {

constexpr int P_STAGES = 6;                          // MMA pipeline ring
constexpr int P_STAGE_TX = A_BYTES + B_HALF;         // 32 KB per CTA per stage
constexpr int Q_STAGES = 10;                         // streaming ring (even: two lanes own a parity each)
constexpr int QT_ROWS = NS / 2;                      // token rows per CTA
constexpr int QT_BYTES = QT_ROWS * KB_BYTES;         // 2 KB
constexpr int Q_STAGE_BYTES = B_HALF + QT_BYTES;     // 18 KB, a multiple of 1024
constexpr int Q_EPI_WARPS = 4;
// Streaming pairs run two pipeline lanes, like the single-CTA kernel's streaming CTAs, with
// the same order of sums: lane p (a TMA thread in each CTA, an MMA thread in the leader)
// takes the K blocks with g % 2 == p of the pair's sequence, in the stages of parity p.
// Lane 0 uses warps 0 and 1, lane 1 the two warps after the streaming epilogue's.
constexpr int Q_PRODUCER1 = 2 + Q_EPI_WARPS, Q_ISSUER1 = Q_PRODUCER1 + 1;
static_assert(Q_ISSUER1 < THREADS / 32, "streaming warps");
constexpr int Q_XPITCH = 17;                         // floats per lane row of the exchange (conflict-free)
constexpr int NBAR_STAGES = Q_STAGES > P_STAGES ? Q_STAGES : P_STAGES;
constexpr unsigned long long DRAIN_NS = 20000000ull;   // waits for work already in flight
// Streaming pairs prefetch their weight boxes this many K blocks ahead of the loads into L2
// (into the pair's next unit near the end of one): a stage waits for both CTAs' copies, so
// the slower of two HBM trips sets its pace, and an L2 hit shortens it (gate/up on the
// prefill mix 4.82 -> 4.49 ms of streaming; the single-CTA streaming role ran slower with the
// same prefetch and does not use it).
constexpr int STREAM_PREFETCH_KB = 16;
constexpr unsigned long long GRACE_NS = 1000000ull;    // rank 1's wait for its own copies after an abort

struct PairSmem {
  // MMA pipeline
  static constexpr int a = 0;
  static constexpr int b = P_STAGES * A_BYTES;
  static constexpr int stage_out = b + P_STAGES * B_HALF;
  static constexpr int x_end = stage_out + EPI_WARPS * STAGE_OUT_BYTES;
  // streaming pairs: Q_STAGES x [128 weight rows | NS/2 token rows], then the SwiGLU
  // exchange between the gate and up warps: float [2 pairs][2 directions][32 lanes][Q_XPITCH]
  static constexpr int q_xch = Q_STAGES * Q_STAGE_BYTES;
  static constexpr int y_end = q_xch + 2 * 2 * 32 * Q_XPITCH * 4;
  static constexpr int common_off = x_end > y_end ? x_end : y_end;
  // common tail: barriers full[S], empty[S], tfull[2], tempty[2], drain[2]; TMEM slot; abort
  // flag; modelled role times; then int bnd[nseg + 1], prefix[nseg + 1], prefix_y[nseg + 1]
  static constexpr int n_bars = 2 * NBAR_STAGES + 6;
  static constexpr int tmem_slot = n_bars * 8;
  static constexpr int abort_flag = tmem_slot + 4;
  static constexpr int costs = abort_flag + 4;
  static constexpr int arrays = 384;
  static size_t bytes(int nseg) {
    return static_cast<size_t>(common_off) + arrays + ((3 * (nseg + 1) * 4 + 15) / 16) * 16 + 1024;
  }
};
static_assert(PairSmem::costs + 8 <= PairSmem::arrays, "common tail header");
static_assert(Q_STAGE_BYTES % 1024 == 0 && P_STAGE_TX % 1024 == 0, "swizzle atoms");

// Modelled time of one pair-unit (relative; all units of a launch have the same K): two
// M-tiles of a segment with more than one M-tile, the single M-tile of a short segment on
// the MMA pipeline (its 256 weight rows stream from HBM behind a shallow ring), and a
// streamed segment.  They set how many pairs stream.  Measured per unit on the prefill
// expert mix with both roles running (gate/up: about 41 us per pipeline unit, 31 us per
// streamed unit on the two streaming lanes).
constexpr float COSTP_MMA = 40.0f, COSTP_SINGLE = 45.0f, COSTP_STREAM = 31.0f;

// ------------------------------------------------------------------ cluster / pair PTX
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t ncluster_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA copy into this CTA's shared memory that completes on `bar`, a barrier of either CTA
// of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                                      uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}
// Bounded wait for work already in flight (after an abort, or at the end).
__device__ __forceinline__ void pdrain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > DRAIN_NS) return;
  }
}
__device__ __forceinline__ void st_remote_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// Wait on a barrier that the partner CTA arrives on (cluster-scope acquire).
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void tc2_commit(uint32_t bar_cluster_addr) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar_cluster_addr)
               : "memory");
}
__device__ __forceinline__ void tc2_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// BF16 x BF16 -> float32, K-major A and B, M = 256 (over the pair), N = n.
__host__ __device__ constexpr uint32_t instr_desc_pair(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(256 >> 4) << 24);
}

// The pair's abort: both CTAs' flags raised (the partner's through its shared memory).
struct PairAbort {
  volatile int* flag;
  uint32_t peer_flag;
  int32_t* dev_status;
  unsigned long long timeout_ns;
  __device__ __forceinline__ void raise() const {
    *flag = 1;
    st_remote_u32(peer_flag, 1u);
    if (dev_status) atomicOr(dev_status, MOE_DEV_PIPELINE_TIMEOUT);
  }
};
// Bounded wait; false if the pair was aborted (this wait timing out, or any role of either CTA).
template <bool CLUSTER>
__device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, const PairAbort& ab) {
  auto tw = [&] { return CLUSTER ? mbar_try_wait_cl(bar, parity) : mbar_try_wait(bar, parity); };
  if (tw()) return true;
  const unsigned long long t0 = globaltimer();
  while (!tw()) {
    if (*ab.flag) return false;
    if (globaltimer() - t0 > ab.timeout_ns) {
      ab.raise();
      return false;
    }
  }
  return true;
}

// Unit u of the MMA pipeline -> segment, N-tile and this CTA's M-tile rows.  The prefix
// counts M-tile pairs, so decode_unit's row0 is the segment start + (pair index) * BM.
__device__ __forceinline__ Unit decode_pair_unit(int u, int n_tiles, const int* bnd, const int* prefix, int nseg,
                                                 int max_tokens, int mgroup, uint32_t crank) {
  Unit w = decode_unit(u, n_tiles, bnd, prefix, nseg, max_tokens, mgroup);
  const int b0 = seg_begin(bnd, w.seg, max_tokens);
  w.row0 = b0 + 2 * (w.row0 - b0) + static_cast<int>(crank) * BM;
  return w;
}

// ------------------------------------------------------------------------ kernel
template <bool SWIGLU>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmBx, const __grid_constant__ CUtensorMap tmBh,
                            const __grid_constant__ CUtensorMap tmBxh, const __grid_constant__ CUtensorMap tmAq,
                            const Args args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* cmn = smem + PairSmem::common_off;
  uint64_t* bars = reinterpret_cast<uint64_t*>(cmn);
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + NBAR_STAGES + s); };
  auto bar_tfull = [&](int b) { return smem_u32(bars + 2 * NBAR_STAGES + b); };
  auto bar_tempty = [&](int b) { return smem_u32(bars + 2 * NBAR_STAGES + 2 + b); };
  const uint32_t bar_drain = smem_u32(bars + 2 * NBAR_STAGES + 4);
  const uint32_t bar_drain1 = smem_u32(bars + 2 * NBAR_STAGES + 5);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cmn + PairSmem::tmem_slot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(cmn + PairSmem::abort_flag);
  float* costs = reinterpret_cast<float*>(cmn + PairSmem::costs);
  const int nseg = args.nseg;
  int* bnd = reinterpret_cast<int*>(cmn + PairSmem::arrays);
  int* prefix = bnd + (nseg + 1);
  int* prefix_y = prefix + (nseg + 1);
  const uint32_t crank = cluster_ctarank();
  const uint32_t peer = crank ^ 1u;
  const bool leader = crank == 0;
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(ncluster_x());

  const int mtok = args.max_tokens;
  if (mtok > 0) {
    for (int i = tid; i < nseg; i += THREADS) bnd[i] = i * mtok + min(max(args.cu[i], 0), mtok);
  } else {
    for (int i = tid; i <= nseg; i += THREADS) bnd[i] = args.cu[i];
  }
  __syncthreads();
  const int n_tiles = SWIGLU ? (args.n_dim / 2) / 128 : (args.n_dim + BN - 1) / BN;
  // per-segment counts -> exclusive prefixes (warp 0): M-tile pairs on the MMA pipeline and
  // streamed segments, plus the modelled time of each role's work
  if (warp == 0) {
    const int chunk = (nseg + 31) / 32;
    const int s0 = min(nseg, lane * chunk), s1 = min(nseg, s0 + chunk);
    auto len = [&](int s) { return max(0, seg_end(bnd, s, mtok) - seg_begin(bnd, s, mtok)); };
    // streaming pays only when every CTA has many units to spread: at least 16 M-tiles x
    // N-tiles per CTA of the grid
    bool stream_on = args.stream != 0;
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
        cy += COSTP_STREAM;
      } else {
        const int m = (l + BM - 1) / BM;
        const int mp = (m + 1) / 2;
        local += mp;
        cx += m == 1 ? COSTP_SINGLE : COSTP_MMA * static_cast<float>(mp);
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
        run += ((l + BM - 1) / BM + 1) / 2;
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
  // pairs [gxp, npairs) stream; every CTA derives the same split from the same counts
  int nyp = 0;
  if (total_y > 0) {
    if (total_units == 0) {
      nyp = npairs;
    } else {
      const float f = costs[1] / (costs[0] + costs[1]);
      nyp = static_cast<int>(f * static_cast<float>(npairs) + 0.5f);
      nyp = min(max(nyp, 1), npairs - 1);
    }
  }
  const int gxp = npairs - nyp;
  const bool y_role = pair >= gxp;
  // MMA-pipeline pairs actually used: the fewest that keep the largest per-pair unit count
  int gxu = gxp;
  if (total_units > 0 && gxp > 0) {
    const int per = (total_units + gxp - 1) / gxp;
    gxu = min(gxp, (total_units + per - 1) / per);
  }
  if (tid == 64) {
    for (int s = 0; s < NBAR_STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull(b), y_role ? 2 : 1);                            // streaming: one per lane
      mbar_init(bar_tempty(b), 2 * (y_role ? Q_EPI_WARPS : EPI_WARPS));   // both CTAs' epilogue warps
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_drain1, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  // the partner's arrivals target this CTA's barriers: both initialise theirs first
  cluster_sync_all();
  // no work for this pair (both CTAs take the same decision): nothing allocated yet
  if (y_role ? pair - gxp >= total_y : pair >= min(total_units, gxu)) return;

  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // both CTAs' tensor memory is allocated before the leader's first MMA
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const PairAbort ab{abort_flag, map_to(smem_u32(cmn + PairSmem::abort_flag), peer), args.dev_status,
                     args.timeout_ns};

  constexpr int KE = 64;  // BF16 K elements per stage
  const int kblocks = args.k_dim / KE;
  const int nst = y_role ? Q_STAGES : P_STAGES;
  const int yi = pair - gxp;
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
  // unit loops of this pair's role: [first, end) with stride
  const int u_first = y_role ? yi : pair;
  const int u_end = y_role ? total_y : total_units;
  const int u_step = y_role ? nyp : gxu;
  const int mgroup = SWIGLU ? MGROUP_GATE_UP / 2 : 0;

  if (warp == 0 || (y_role && warp == Q_PRODUCER1)) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    // (streaming: lane p = 0, 1 fills the stages of parity p)
    if (lane == 0) {
      const uint32_t lp = warp == 0 ? 0u : 1u;
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
      int stage = 0;
      uint32_t phase = 0, armed = 0, last_parity = 0, g = 0;
      bool ok = true;
      uint64_t wpol;
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(wpol));
      const uint32_t lead_full = map_to(bar_full(0), 0);
      for (int u = u_first; ok && u < u_end; u += u_step) {
        int seg, nt, row0;
        if (y_role) {
          y_unit(u, seg, nt);
          row0 = seg_begin(bnd, seg, mtok) + QT_ROWS * static_cast<int>(crank);
        } else {
          const Unit w = decode_pair_unit(u, n_tiles, bnd, prefix, nseg, mtok, mgroup, crank);
          seg = w.seg;
          nt = w.nt;
          row0 = w.row0;
        }
        const bool extra = seg >= args.num_w;
        const int wbase = extra ? 0 : seg * args.n_dim;
        // streaming: this CTA's weight boxes of this unit and of its next one, prefetched into
        // L2 STREAM_PREFETCH_KB K blocks ahead of the loads
        const CUtensorMap* pm = nullptr;
        const CUtensorMap* npm = nullptr;
        int p0 = 0, p1 = -1, n0 = -1, n1 = -1;
        if (y_role) {
          pm = SWIGLU ? (extra ? &tmBxh : &tmBh) : (extra ? &tmBx : &tmB);
          p0 = SWIGLU ? wbase + nt * 128 + 64 * static_cast<int>(crank) : wbase + nt * BN + 128 * static_cast<int>(crank);
          p1 = SWIGLU ? p0 + args.n_dim / 2 : -1;
          if (u + u_step < u_end) {
            int s2, nt2;
            y_unit(u + u_step, s2, nt2);
            const bool x2 = s2 >= args.num_w;
            const int wb2 = x2 ? 0 : s2 * args.n_dim;
            npm = SWIGLU ? (x2 ? &tmBxh : &tmBh) : (x2 ? &tmBx : &tmB);
            n0 = SWIGLU ? wb2 + nt2 * 128 + 64 * static_cast<int>(crank) : wb2 + nt2 * BN + 128 * static_cast<int>(crank);
            n1 = SWIGLU ? n0 + args.n_dim / 2 : -1;
          }
        }
        for (int kb = 0; kb < kblocks; ++kb, ++g) {
          if (y_role && (g & 1u) != lp) {   // the other lane's K block
            if (++stage == nst) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          if (y_role) {
            const int pk = kb + STREAM_PREFETCH_KB;
            if (pk < kblocks) {
              tma_prefetch_2d(pm, pk * KE, p0);
              if (p1 >= 0) tma_prefetch_2d(pm, pk * KE, p1);
            } else if (n0 >= 0 && pk - kblocks < kblocks) {
              tma_prefetch_2d(npm, (pk - kblocks) * KE, n0);
              if (n1 >= 0) tma_prefetch_2d(npm, (pk - kblocks) * KE, n1);
            }
          }
          if (!pwait<false>(bar_empty(stage), phase ^ 1, ab)) {
            ok = false;
            break;
          }
          armed |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          // every copy of the stage completes on the leader's full barrier, armed there with
          // the bytes of both CTAs
          const uint32_t fb = lead_full + 8u * stage;
          if (leader) mbar_expect_tx(bar_full(stage), 2 * (y_role ? Q_STAGE_BYTES : P_STAGE_TX));
          if (y_role) {
            const uint32_t sw = sbase + stage * Q_STAGE_BYTES;
            if (SWIGLU) {
              // 64 gate rows and the matching 64 up rows of this CTA's output columns
              const CUtensorMap* mh = extra ? &tmBxh : &tmBh;
              const int g0 = wbase + nt * 128 + 64 * static_cast<int>(crank);
              tma_load_2d_pair_hint(sw, mh, kb * KE, g0, fb, wpol);
              tma_load_2d_pair_hint(sw + B_HALF / 2, mh, kb * KE, g0 + args.n_dim / 2, fb, wpol);
            } else {
              const CUtensorMap* mb = extra ? &tmBx : &tmB;
              tma_load_2d_pair_hint(sw, mb, kb * KE, wbase + nt * BN + 128 * static_cast<int>(crank), fb, wpol);
            }
            tma_load_2d_pair(sw + B_HALF, &tmAq, kb * KE, row0, fb);
          } else {
            const CUtensorMap* mb = extra ? &tmBx : &tmB;
            const int rb = SWIGLU ? wbase + (crank ? args.n_dim / 2 : 0) + nt * 128
                                  : wbase + nt * BN + 128 * static_cast<int>(crank);
            tma_load_2d_pair(sbase + PairSmem::a + stage * A_BYTES, &tmA, kb * KE, row0, fb);
            tma_load_2d_pair(sbase + PairSmem::b + stage * B_HALF, mb, kb * KE, rb, fb);
          }
          if (++stage == nst) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // copies still in flight land before this CTA's shared memory goes away: the leader
        // sees both CTAs' copies of every stage it armed complete on its barriers; rank 1
        // cannot observe its own, and gives them a grace period
        if (leader) {
          for (int s = 0; s < nst; ++s)
            if (armed & (1u << s)) pdrain(bar_full(s), (last_parity >> s) & 1u);
        } else {
          const unsigned long long t0 = globaltimer();
          while (globaltimer() - t0 < GRACE_NS) {
          }
        }
      } else {
        // every stage this CTA filled has been released by the leader's MMAs: no MMA reads
        // this CTA's shared memory any more and no commit is still on its way here
        for (int s = 0; s < nst; ++s)
          if (armed & (1u << s)) pdrain(bar_empty(s), (last_parity >> s) & 1u);
      }
    }
  } else if (warp == 1 || (y_role && warp == Q_ISSUER1)) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer (leader; streaming:
      // lane p = 0, 1 consumes the stages of parity p)
      const uint32_t lp = warp == 1 ? 0u : 1u;
      const uint32_t drain = lp == 0 ? bar_drain : bar_drain1;
      const uint32_t idesc = instr_desc_pair(y_role ? NS : BN);
      const int acc_cols = y_role ? NS : BN;
      int stage = 0, buf = 0;
      uint32_t phase = 0, tphase = 0, g = 0;
      bool ok = true;
      for (int u = u_first; ok && u < u_end; u += u_step) {
        for (int kb = 0; kb < kblocks; ++kb, ++g) {
          if (kb == 0) {
            if (!pwait<true>(bar_tempty(buf), tphase ^ 1, ab)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (y_role && (g & 1u) != lp) {   // the other lane's K block
            if (++stage == nst) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          if (!pwait<false>(bar_full(stage), phase, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t sa, sb;
          if (y_role) {
            sa = sbase + stage * Q_STAGE_BYTES;     // weights: the M operand
            sb = sa + B_HALF;                       // the segment's rows: the N operand
          } else {
            sa = sbase + PairSmem::a + stage * A_BYTES;
            sb = sbase + PairSmem::b + stage * B_HALF;
          }
          // streaming pairs: even and odd K blocks accumulate apart (columns [2 NS b, +NS) and
          // [2 NS b + NS, +NS)) and the epilogue adds the two sums, the order of the single-CTA
          // kernel's two streaming lanes (k_dim % 128 == 0: an even K-block count)
          const bool split = y_role;
          const uint32_t dt = y_role ? tmem_base + buf * (2 * NS) + ((split && (kb & 1)) ? NS : 0) : tmem_base + buf * acc_cols;
          const int kfirst = split ? (kb >> 1) : kb;
#pragma unroll
          for (int k = 0; k < KB_BYTES / 32; ++k)
            tc2_mma(dt, smem_desc(sa + 32 * k), smem_desc(sb + 32 * k), idesc, (kfirst | k) != 0);
          tc2_commit(bar_empty(stage));
          tc2_commit(map_to(bar_empty(stage), peer));
          if (++stage == nst) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc2_commit(bar_tfull(buf));   // streaming: one of the two arrivals
        tc2_commit(map_to(bar_tfull(buf), peer));
        if (++buf == 2) {
          buf = 0;
          tphase ^= 1;
        }
      }
      if (!ok) {
        tc2_commit(drain);  // arrives once every MMA this thread issued has completed
        pdrain(drain, 0);
      }
    }
  } else if (!y_role) {
    // ------------------------------------------------------------ epilogue (MMA pipeline)
    const int q = warp & 3;               // TMEM subpartition this warp may access
    const int half = (warp - 2) >> 2;     // which half of the tile's columns
    const int r_in_tile = 32 * q + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t tempty_lead = map_to(bar_tempty(0), 0);
    int buf = 0;
    uint32_t tphase = 0;
    const int out_cols = SWIGLU ? args.n_dim / 2 : args.n_dim;
    uint8_t* stage_out = smem + PairSmem::stage_out;
    for (int u = u_first; u < u_end; u += u_step) {
      const Unit w = decode_pair_unit(u, n_tiles, bnd, prefix, nseg, mtok, mgroup, crank);
      const int row = w.row0 + r_in_tile;
      const bool row_ok = row < w.row_end;
      const int col0 = SWIGLU ? w.nt * 128 + 64 * half : w.nt * BN + 128 * half;
      const bool cols_ok = col0 < out_cols;
      float acc[128];
      if (!pwait<true>(bar_tfull(buf), tphase, ab)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + lane_addr + buf * BN;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int tcol = SWIGLU ? (c < 2 ? 64 * half + 32 * c : 128 + 64 * half + 32 * (c - 2)) : 128 * half + 32 * c;
        uint32_t r[32];
        tmem_ld32(tb + tcol, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[32 * c + i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(bar_tempty(buf));
        else
          mbar_arrive_remote(tempty_lead + 8u * buf);
      }
      if (++buf == 2) {
        buf = 0;
        tphase ^= 1;
      }
      if (SWIGLU) {
        if (row_ok && cols_ok) {
          float h[64];
#pragma unroll
          for (int i = 0; i < 64; ++i) h[i] = silu(acc[i]) * acc[64 + i];
          store_h_bf16(h, static_cast<uint16_t*>(args.out) + (size_t)row * out_cols + col0);
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
      }
    }
  } else if (warp < 2 + Q_EPI_WARPS) {
    // ------------------------------------------------------------ epilogue (streaming pairs)
    // warp w reads TMEM lanes 32 (w % 4).. = this CTA's weight rows; 32 token columns each
    const int q = warp & 3;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t tempty_lead = map_to(bar_tempty(0), 0);
    const int out_cols = SWIGLU ? args.n_dim / 2 : args.n_dim;
    float* xch = reinterpret_cast<float*>(smem + PairSmem::q_xch);
    int buf = 0;
    uint32_t tphase = 0;
    for (int v = yi; v < total_y; v += nyp) {
      int seg, nt;
      y_unit(v, seg, nt);
      const int row0 = seg_begin(bnd, seg, mtok), row_end = seg_end(bnd, seg, mtok);
      const bool ok = pwait<true>(bar_tfull(buf), tphase, ab);
      // the four warps leave together (their exchange below uses a named barrier)
      if (bar_red_or(2, 32 * Q_EPI_WARPS, !ok)) break;
      tc_fence_after();
      uint32_t d[NS];
      tmem_ld32(tmem_base + lane_addr + buf * (2 * NS), d);
      tmem_wait_ld();
      {
        uint32_t e[NS];
        tmem_ld32(tmem_base + lane_addr + buf * (2 * NS) + NS, e);
        tmem_wait_ld();
#pragma unroll
        for (int n = 0; n < NS; ++n) d[n] = __float_as_uint(__fadd_rn(__uint_as_float(d[n]), __uint_as_float(e[n])));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(bar_tempty(buf));
        else
          mbar_arrive_remote(tempty_lead + 8u * buf);
      }
      if (++buf == 2) {
        buf = 0;
        tphase ^= 1;
      }
      const int rows = min(row_end - row0, NS);
      if (SWIGLU) {
        // lanes 0-63: gate rows of output columns 128 nt + 64 rank + j; lanes 64-127: the
        // matching up rows.  Gate warp (q < 2) computes tokens [0, NS/2), up warp (q + 2)
        // tokens [NS/2, NS), each taking the other's half through shared memory.
        const bool gate = q < 2;
        const int pq = q & 1;
        float* to_up = xch + ((pq * 2 + 0) * 32 + lane) * Q_XPITCH;     // gate values of tokens NS/2..
        float* to_gate = xch + ((pq * 2 + 1) * 32 + lane) * Q_XPITCH;   // up values of tokens 0..
#pragma unroll
        for (int n = 0; n < NS / 2; ++n) {
          if (gate)
            to_up[n] = __uint_as_float(d[NS / 2 + n]);
          else
            to_gate[n] = __uint_as_float(d[n]);
        }
        asm volatile("bar.sync 2, %0;" ::"r"(32 * Q_EPI_WARPS) : "memory");
        const int col = nt * 128 + 64 * static_cast<int>(crank) + 32 * pq + lane;
        uint16_t* dst = static_cast<uint16_t*>(args.out) + (size_t)row0 * out_cols + col;
        if (gate) {
#pragma unroll
          for (int n = 0; n < NS / 2; ++n)
            if (n < rows) dst[(size_t)n * out_cols] = f32_to_bf16(silu(__uint_as_float(d[n])) * to_gate[n]);
        } else {
#pragma unroll
          for (int n = 0; n < NS / 2; ++n)
            if (NS / 2 + n < rows)
              dst[(size_t)(NS / 2 + n) * out_cols] = f32_to_bf16(silu(to_up[n]) * __uint_as_float(d[NS / 2 + n]));
        }
      } else {
        const int col = nt * BN + 128 * static_cast<int>(crank) + 32 * q + lane;
        if (col < out_cols) {
          uint16_t* dst = static_cast<uint16_t*>(args.out) + (size_t)row0 * out_cols + col;
#pragma unroll
          for (int n = 0; n < NS; ++n) {
            if (n < rows) {
              float vv = __uint_as_float(d[n]);
              if (args.row_scale) vv = __fmul_rn(vv, args.row_scale[row0 + n]);
              dst[(size_t)n * out_cols] = f32_to_bf16(vv);
            }
          }
        }
      }
    }
  }
  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // neither CTA frees its memory while the partner may still reach it
  tc_fence_after();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
}

// ---------------------------------------------------------------------- host side
template <bool SWIGLU>
static moe_status_t launch_2sm_impl(const CUtensorMap* maps, const Args& args_in, long long max_pair_units,
                                    bool stream_ok, cudaStream_t s) {
  auto kern = grouped_gemm_2sm_kernel<SWIGLU>;
  static std::atomic<unsigned long long> attr_done{0};
  if (!once_per_device(attr_done, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX) == cudaSuccess &&
               cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) == cudaSuccess;
      }))
    return MOE_ERR_CUDA;
  Args args = args_in;
  const size_t smem = PairSmem::bytes(args.nseg);
  if (smem > (size_t)SMEM_MAX) return MOE_ERR_ARG;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 2;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  // pairs that fit on the GPU at once (clusters stay within a GPC), looked up per device
  static std::atomic<int> max_pairs_cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  int max_pairs = max_pairs_cache[dev & 63].load(std::memory_order_relaxed);
  if (max_pairs <= 0) {
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) return MOE_ERR_CUDA;
    max_pairs = n;
    max_pairs_cache[dev & 63].store(n, std::memory_order_relaxed);
  }
  const int pairs = static_cast<int>(std::min<long long>(std::min(max_pairs, num_sms() / 2), max_pair_units));
  if (pairs < 1) return MOE_ERR_UNSUPPORTED;
  args.stream = stream_ok && 2 * pairs >= 16 ? 1 : 0;
  cfg.gridDim = dim3(2 * pairs);
  if (cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], args) != cudaSuccess)
    return MOE_ERR_CUDA;
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

// BF16 grouped GEMM on CTA pairs: tensor maps of A (128-row box), the routed weights and
// the extra segment's weights (128-row boxes and 64-row boxes), and A again with NS/2-row
// boxes for the streaming pairs.
moe_status_t launch_2sm(const void* a, int rows_cap, int k_dim, int n_dim, const void* w, int num_w,
                        const void* w_extra, bool swiglu, const Args& args, bool stream_ok, cudaStream_t s) {
  CUtensorMap maps[6];
  if (!make_map(&maps[0], a, false, k_dim, rows_cap)) return MOE_ERR_CUDA;
  const void* wb = num_w > 0 ? w : w_extra;
  const uint64_t wrows = num_w > 0 ? (uint64_t)num_w * n_dim : (uint64_t)n_dim;
  if (!make_map(&maps[1], wb, false, k_dim, wrows)) return MOE_ERR_CUDA;
  if (!make_map(&maps[3], wb, false, k_dim, wrows, 64)) return MOE_ERR_CUDA;
  if (w_extra) {
    if (!make_map(&maps[2], w_extra, false, k_dim, n_dim)) return MOE_ERR_CUDA;
    if (!make_map(&maps[4], w_extra, false, k_dim, n_dim, 64)) return MOE_ERR_CUDA;
  } else {
    maps[2] = maps[1];
    maps[4] = maps[3];
  }
  if (!make_map(&maps[5], a, false, k_dim, rows_cap, QT_ROWS)) return MOE_ERR_CUDA;
  const int n_tiles = swiglu ? (n_dim / 2) / 128 : (n_dim + BN - 1) / BN;
  // at most (M-tiles + segments) / 2 + segments pairs of M-tiles per N-tile
  const long long m_tiles = (long long)(rows_cap + BM - 1) / BM + args.nseg;
  const long long max_pair_units = (m_tiles / 2 + args.nseg) * n_tiles;
  return swiglu ? launch_2sm_impl<true>(maps, args, max_pair_units, stream_ok, s)
                : launch_2sm_impl<false>(maps, args, max_pair_units, stream_ok, s);
}

}  // namespace gg
}  // namespace moe
