/*
 * moe.h -- C ABI of libmoe: the single-GPU Mixture-of-Experts layer hot path on GB300
 * (sm_103a): route -> permute -> grouped GEMM (gate/up + SwiGLU, down) -> combine.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named in a signature are DEVICE pointers unless the comment says "host".
 *   All buffers are owned by the caller; the library never allocates, frees, copies to
 *   the host or synchronises.  Every call only enqueues kernels on `stream` (a
 *   cudaStream_t passed as void*; NULL = the legacy default stream) and returns, so a
 *   sequence of calls can be captured in a CUDA graph.
 * - Host-side argument errors (bad sizes, null required pointers, a workspace that is
 *   too small) are detected before anything is enqueued and returned as a moe_status_t;
 *   nothing is launched in that case.  MOE_ERR_CUDA reports a failed launch.
 * - Data errors found on the device (an expert id outside [-1, E), a verification
 *   mismatch, a pipeline wait that ran out of time) never trap: they OR a bit into the
 *   caller's int32 `dev_status` word (device memory, zeroed by the caller, sticky).
 * - Tensors are dense and row-major.  BF16 is passed as uint16_t bit patterns, FP8 E4M3
 *   ("e4m3fn": bias 7, max 448, no infinities) as uint8_t codes.
 * - T tokens (rows of the batch, possibly a padded bucket), H hidden size, I expert
 *   intermediate size, E routed experts, K experts per token.  H and I must be
 *   multiples of 128 (the 128-wide tile constraint the MoonEP page validates at layout
 *   construction), 1 <= K <= min(E, 32), E <= 1024.
 *
 * Sources (four pull-request pages):
 *   [MegaMoE]  "Add MoE dispatch/combine fake quantization for vLLM's DeepGEMM Mega-MoE"
 *   [DeepEP]   "[Kernel] DeepEP dispatch-combine kernel integration"
 *   [MoonEP]   "[Distributed][MoonEP] BF16 integration of MoonEP balanced EP backend"
 *   [Scratch]  "[Bugfix][MoE] Size the permute scratch from its inputs"
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_ARG = 1,          /* bad size or null required pointer (host-side, nothing launched) */
  MOE_ERR_WORKSPACE = 2,    /* workspace smaller than the size query returns */
  MOE_ERR_UNSUPPORTED = 3,  /* valid request the library does not implement */
  MOE_ERR_CUDA = 4          /* a CUDA runtime call or launch failed */
} moe_status_t;

typedef enum { MOE_BF16 = 0, MOE_E4M3 = 1 } moe_dtype_t;
/* ORed into the dtype argument of moe_grouped_gemm, _ex, _batched and _combine: w and
 * w_extra are in the tile layout of moe_pack_weights (ABI 6). */
#define MOE_W_TILED 0x100
typedef enum { MOE_EPI_NONE = 0, MOE_EPI_SWIGLU = 1 } moe_epilogue_t;

/* Bits of the device status word. */
#define MOE_DEV_BAD_EXPERT 1        /* an expert id outside [-1, E): slot treated as padding */
#define MOE_DEV_VERIFY_MISMATCH 2   /* moe_combine_verify found an element that differs */
#define MOE_DEV_PIPELINE_TIMEOUT 4  /* a GEMM pipeline wait gave up; its output is invalid */
#define MOE_DEV_OVERFLOW 8          /* batched layout: a segment received more than max_tokens
                                       rows; the slots past max_tokens were dropped */

/* Version of this ABI (bumped on any signature change; 2 added the weight_in_down and
 * dispatch fake-quant options, 3 the batched expert layout, 4 the NVFP4 combine
 * and dispatch fake-quant (moe_combine_nvfp4, the dispatch_format arguments,
 * moe_layer_desc_t.combine_fq_format / dispatch_fq_format), 5 moe_grouped_gemm_pairs,
 * 6 the tiled weight layout: moe_pack_weights, MOE_W_TILED, moe_layer_desc_t.weight_tiles). */
int moe_abi_version(void);
/* Static, human-readable name of a status code. */
const char* moe_status_string(moe_status_t s);

/* ---------------------------------------------------------------------------- route
 * Router: softmax over E, top-K, renormalise over the K chosen.
 * [DeepEP] passes per-token topk_weights / topk_ids into dispatch and [MoonEP] works with
 * [T, K] expert ids; neither page defines the router function, so this takes the plain
 * softmax -> top-k -> renormalise reading.
 *   logits     float32 [T, E], finite.
 *   num_tokens nullable device int32 scalar n: rows t >= n are padding of a receive
 *              bucket ([Scratch]: power-of-two buckets) and get ids -1, weights 0.  NULL
 *              means all T rows are tokens.  Read on the device, so a captured graph can
 *              be replayed with a different n.
 *   topk_idx   out int32 [T, K]: expert ids in descending logit order, ties to the lower
 *              id (bit-exact: chosen on the float32 logits).
 *   topk_w     out float32 [T, K]: w_k = e^{l_k - l_0} / sum_j e^{l_j - l_0}, computed in
 *              float32 with expf (the full softmax denominator cancels).
 * Errors: MOE_ERR_ARG if T < 0, E < 1 or E > 1024, K < 1, K > min(E, 32), a null
 * pointer with T > 0. */
moe_status_t moe_route_topk(const float* logits, int T, int E, int K, const int32_t* num_tokens,
                            int32_t* topk_idx, float* topk_w, void* stream);

/* -------------------------------------------------------------------------- permute
 * Dispatch into the expert-major layout: a stable counting sort of the valid
 * (token, slot) pairs by expert id ([MoonEP]: after dispatch the rows arrive grouped by
 * expert, [NvS, H] plus cu_seqlens; [DeepEP]: moe_permute_unpermute), then a gather of each
 * row's token.  Flat slot s = t*K + k; segment e holds the slots with topk_idx == e in
 * ascending s.  topk_idx == -1 marks padding ([MegaMoE]: valid = topk_idx >= 0): no row.
 *
 * with_shared = 1 appends segment E for the shared expert: every token with at least
 * one valid slot, ascending t, source index T*K + t ([MegaMoE]: the fused shared
 * expert's slot; here it is one more dense segment of the same grouped GEMM).
 *
 * Sizes come from the inputs, never from a model config ([Scratch]: the bound is the
 * rows times experts_per_token actually received):
 *   cap = T*K + (with_shared ? T : 0)   rows of xp / src_row
 *   nseg = E + with_shared              segments
 *   x          BF16 [T, H] token activations.
 *   out_dtype  MOE_BF16: xp is BF16 [cap, H], exact copies of the rows.
 *              MOE_E4M3: xp is E4M3 [cap, H] and xp_scales float32 [cap, H/128]: each
 *              row quantised per 1x128 block on the fly (s = amax/448, 1 if amax is 0;
 *              q = e4m3_rn_satfinite(x / s)), the internal FP8 quantisation the [DeepEP]
 *              low-latency dispatch applies to BF16 tokens.
 *   cu_seqlens out int32 [nseg + 1], cu[0] = 0, cu[nseg] = rows written (N).
 *   src_row    out int32 [cap]: source index of each row (t*K+k, or T*K+t for a shared
 *              row); -1 for rows >= N.
 *   inv_map    out int32 [T, K]: row of each slot, -1 for padding.
 *   shared_map out int32 [T] (required iff with_shared): shared row of each token, or -1.
 *   ws         scratch of at least moe_permute_workspace_bytes(T, K, E, with_shared) bytes,
 *              256-byte aligned; it holds index metadata only ([Scratch]: the permute
 *              scratch carries no hidden states), no state kept between calls.
 *   dev_status nullable; MOE_DEV_BAD_EXPERT is ORed in for ids outside [-1, E).
 * Rows of xp at or past N are not written.
 * Errors: MOE_ERR_ARG for bad sizes / null pointers, MOE_ERR_WORKSPACE if ws_bytes is short. */
size_t moe_permute_workspace_bytes(int T, int K, int E, int with_shared);
moe_status_t moe_permute(const int32_t* topk_idx, int T, int K, int E, int with_shared,
                         const uint16_t* x, int H, moe_dtype_t out_dtype, void* xp, float* xp_scales,
                         int32_t* cu_seqlens, int32_t* src_row, int32_t* inv_map, int32_t* shared_map,
                         void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* moe_permute for callers that cannot allocate device memory.  (The pages have no
 * counterpart: this is an addition of this library.)  Some callers may not call cudaMalloc:
 * plugins inside an inference engine that owns every device allocation, code running while
 * its stream is captured into a CUDA graph, serving paths with a fixed memory budget.  This
 * variant takes no workspace: its index scratch is a static device array of
 * moe_permute_noalloc_max_scratch_bytes() bytes (1 MiB) that every GPU loading the library
 * holds until the process exits.  Arguments and outputs are those of moe_permute.
 * - Shapes whose scratch (moe_permute_workspace_bytes) exceeds that maximum are rejected
 *   with MOE_ERR_WORKSPACE before anything is launched (e.g. E = 256 with a shared
 *   expert fits T up to about 65000 tokens; E = 1024 about 16000).
 * - The first call on each device looks up the array's device address (cudaGetSymbolAddress
 *   with that device current) and caches it with the device's current context; make that
 *   first call before any stream capture begins.  After a device reset the next call sees
 *   a new context and looks the address up again (also outside a capture).  MOE_ERR_CUDA
 *   if the lookup fails.
 * - All calls on a device share the array.  Nothing in it needs to start at zero, but calls
 *   whose kernels overlap on the GPU (unordered streams) race on it; order them. */
size_t moe_permute_noalloc_max_scratch_bytes(void);
moe_status_t moe_permute_noalloc(const int32_t* topk_idx, int T, int K, int E, int with_shared,
                                 const uint16_t* x, int H, moe_dtype_t out_dtype, void* xp, float* xp_scales,
                                 int32_t* cu_seqlens, int32_t* src_row, int32_t* inv_map,
                                 int32_t* shared_map, int32_t* dev_status, void* stream);

/* moe_permute with two options (ABI 2; dispatch_format ABI 4):
 *   dispatch_scale nullable device float32 s: dispatch fake-quant ([MegaMoE]: the dispatch
 *              quantiser fake-quantises the tokens the routed experts receive, with a
 *              calibrated or constant global scale; the shared expert must not see them,
 *              so the shared rows keep the original x).  BF16 output only
 *              (MOE_ERR_UNSUPPORTED for E4M3, whose rows are quantised anyway).
 *   dispatch_format 0: E4M3 -- routed rows become bf16(float(e4m3_rn_satfinite(x * s)) / s),
 *              float32 steps.  1: NVFP4 ([MegaMoE]'s other dispatch unit; s is the
 *              per-tensor scale g = 448 * 6 / amax) -- per 16 consecutive columns the
 *              moe_combine_nvfp4 step applied to x, rounded to BF16.  Else MOE_ERR_ARG.
 *   topk_w / row_weights  nullable; with both given, row_weights float32 [cap] receives each
 *              row's router weight (topk_w[t, k] of its slot, 1 for a shared row), for a down
 *              projection that applies the weights itself (moe_grouped_gemm_ex row_scale).
 * Everything else as moe_permute. */
moe_status_t moe_permute_ex(const int32_t* topk_idx, int T, int K, int E, int with_shared,
                            const uint16_t* x, int H, moe_dtype_t out_dtype, void* xp, float* xp_scales,
                            int32_t* cu_seqlens, int32_t* src_row, int32_t* inv_map, int32_t* shared_map,
                            void* ws, size_t ws_bytes, int32_t* dev_status, const float* dispatch_scale,
                            int dispatch_format, const float* topk_w, float* row_weights, void* stream);

/* Calibration of the dispatch scale: amax = max(amax, max |x|) over a BF16 tensor of n
 * elements (16-byte aligned).  amax is a device float32 the caller zeroes; then
 * moe_fq_scale_from_amax gives 448 / amax. */
moe_status_t moe_amax_bf16(const uint16_t* x, size_t n, float* amax, void* stream);

/* ---------------------------------------------------------------------- FP8 quantise
 * Activation quantisation per 1x128 block ([DeepEP]: FP8 dispatch of "tokens, and
 * scales" dequantised at the receiver):  x BF16 [rows, cols] -> q E4M3 [rows, cols],
 * scales float32 [rows, cols/128]; s = amax/448 (1 if that is not positive),
 * q = e4m3_rn_satfinite(x / s), divisions in IEEE float32.  cols % 128 == 0. */
moe_status_t moe_quantize_act_fp8(const uint16_t* x, int rows, int cols, uint8_t* q, float* scales,
                                  void* stream);
/* Weight quantisation per 128x128 block ([DeepEP] test: block_n x block_k weight tiles):
 * w BF16 [mats, rows, cols] -> q E4M3 same shape, scales float32
 * [mats, rows/128, cols/128], same rule as above.  rows % 128 == cols % 128 == 0.
 * A one-time weight-preparation call (outside the layer). */
moe_status_t moe_quantize_weight_fp8(const uint16_t* w, int mats, int rows, int cols, uint8_t* q,
                                     float* scales, void* stream);

/* ---------------------------------------------------------------------- grouped GEMM
 * Grouped GEMM over the cu_seqlens segments ([MoonEP]: the gate, up and down projections
 * run as grouped matmuls over the segments, and a segment with no rows costs nothing).
 * For each segment s and each row r in [cu[s], cu[s+1]):
 *     acc[r, n] = sum_k a[r, k] * W_s[n, k]      (FP32 accumulation, tensor cores)
 * W_s = w + s*n_dim*k_dim for s < num_w, and w_extra for s == num_w (the shared expert).
 *   a          BF16 or E4M3 [rows_cap, k_dim]; a_scales float32 [rows_cap, k_dim/128] for E4M3.
 *   w          [num_w, n_dim, k_dim] (K-major rows) of dtype; w_scales float32
 *              [num_w, n_dim/128, k_dim/128] for E4M3 (dequantised value = q * s).
 *   w_extra    nullable [n_dim, k_dim]; w_extra_scales [n_dim/128, k_dim/128] for E4M3.
 *   epilogue   MOE_EPI_NONE:   out BF16 [rows_cap, n_dim] = bf16_rn(acc).
 *              MOE_EPI_SWIGLU: n_dim = 2*I, weight rows [0, I) are the gate and [I, 2I) the
 *              up projection ([DeepEP]: w1 with 2n rows); h = silu(g) * u with
 *              silu(z) = z / (1 + e^-z), out [rows_cap, I] = bf16_rn(h) for BF16, or
 *              E4M3 codes with out_scales float32 [rows_cap, I/128] (1x128 blocks, the
 *              rule of moe_quantize_act_fp8) for E4M3.
 *   num_segments <= num_w + (w_extra != NULL).  Rows of out outside every segment are not
 *   written.  k_dim % 128 == 0, n_dim % 128 == 0 (SwiGLU: I % 128 == 0).
 *   dev_status nullable; MOE_DEV_PIPELINE_TIMEOUT if a pipeline wait gave up.
 * Errors: MOE_ERR_ARG for bad sizes / null pointers / misaligned pointers (a, w and out
 * must be 16-byte aligned). */
moe_status_t moe_grouped_gemm(const void* a, const float* a_scales, const int32_t* cu_seqlens,
                              int num_segments, int rows_cap, int k_dim, int n_dim,
                              const void* w, const float* w_scales, int num_w,
                              const void* w_extra, const float* w_extra_scales,
                              moe_dtype_t dtype, moe_epilogue_t epilogue, void* out, float* out_scales,
                              int32_t* dev_status, void* stream);

/* moe_grouped_gemm with a per-row output scale (ABI 2): row_scale nullable float32
 * [rows_cap]; with MOE_EPI_NONE the float32 accumulator of out row r is multiplied by
 * row_scale[r] before the BF16 rounding.  This applies the router weights inside the
 * down projection ([MoonEP]: route weights applied in the expert computation, so the
 * combine only sums); rejected (MOE_ERR_ARG) with MOE_EPI_SWIGLU. */
moe_status_t moe_grouped_gemm_ex(const void* a, const float* a_scales, const int32_t* cu_seqlens,
                                 int num_segments, int rows_cap, int k_dim, int n_dim,
                                 const void* w, const float* w_scales, int num_w,
                                 const void* w_extra, const float* w_extra_scales,
                                 moe_dtype_t dtype, moe_epilogue_t epilogue, void* out, float* out_scales,
                                 int32_t* dev_status, const float* row_scale, void* stream);

/* moe_grouped_gemm_ex for BF16 computed on pairs of SMs (ABI 5): each 256-row M tile is
 * split over the two CTAs of a 2-CTA cluster, which share one 256-wide weight tile through
 * the 2-SM tensor-core MMA ([MoonEP] "Purpose": the gate, up and down grouped matmuls over
 * the cu_seqlens segments).  Same arguments, layouts and results as moe_grouped_gemm_ex with
 * dtype MOE_BF16 (the output is identical bit for bit); segments of at most 32 rows run on
 * weight-streaming pairs when the launch has many units.  Which of the two is faster depends
 * on the segment mix: on a mix of a few large and many tiny segments (the Zipf-routed prefill
 * batch) this one is slower, on dense segments of a few hundred rows it is as fast or faster;
 * moe_layer_forward uses moe_grouped_gemm_ex.  Errors as moe_grouped_gemm_ex. */
moe_status_t moe_grouped_gemm_pairs(const void* a, const int32_t* cu_seqlens, int num_segments, int rows_cap,
                                    int k_dim, int n_dim, const void* w, int num_w, const void* w_extra,
                                    moe_epilogue_t epilogue, void* out, int32_t* dev_status,
                                    const float* row_scale, void* stream);

/* Tiled weight layout (ABI 6; an addition of this library, the pages have no counterpart).
 * The grouped GEMM reads a weight matrix as boxes of 128 rows x 128 bytes of K (64 BF16 or
 * 128 E4M3 elements); in the row-major layout such a box is 128 pieces of 128 bytes, one
 * per row, a row (k_dim elements) apart, and a segment of a few rows streams its weights
 * as a sequence of such scattered pieces.  moe_pack_weights writes a copy of the weights
 * in which every box is 16 contiguous KB:
 *   w        [E, N, K] (K-major rows) of dtype, N % 128 == 0, K % 128 == 0.
 *   w_tiled  out, the same number of bytes: box (e, nb, kb) -- rows [128 nb, 128 nb + 128)
 *            of matrix e, bytes [128 kb, 128 kb + 128) of each row -- at byte offset
 *            ((e * (N / 128) + nb) * (K * esize / 128) + kb) * 16384, its 128 rows of
 *            128 bytes in order (esize = 2 for BF16, 1 for E4M3).
 * The shared expert's matrix is packed the same way with E = 1.  The E4M3 weight scales
 * keep their layout.  A one-time preparation of model weights; asynchronous on stream.
 * Errors: MOE_ERR_ARG for bad sizes, a null or misaligned (16 bytes) pointer, or
 * overlapping w and w_tiled. */
moe_status_t moe_pack_weights(const void* w, int E, int N, int K, moe_dtype_t dtype, void* w_tiled, void* stream);

/* A grouped GEMM call whose dtype argument carries MOE_W_TILED (moe_grouped_gemm, _ex,
 * _batched, _combine) reads w and w_extra in this layout; every other argument and the
 * results, bit for bit, are those of the row-major call.  On the Zipf-routed prefill batch
 * the weight stream of the many experts with a few rows is faster from contiguous boxes.
 * Errors: those of the call, and MOE_ERR_ARG when num_w * n_dim * k_dim / (64 BF16 or 128
 * E4M3 elements) exceeds 2^31 - 1; moe_grouped_gemm_pairs has no dtype argument and reads
 * row-major weights only. */

/* ------------------------------------------------------------ batched expert layout
 * The expert-batched activation format ([DeepEP]: the low-latency dispatch hands the
 * experts one fixed block of rows per expert, 3-D [E, max_tokens, H], while the
 * high-throughput dispatch produces the 2-D contiguous layout above; the experts' kernel has
 * to know which format it gets).  Segment s owns rows [s*max_tokens, (s+1)*max_tokens) of
 * a [nseg * max_tokens, H] buffer; its first masked_m[s] rows are real, the rest padding
 * that no call reads or writes.
 *
 * moe_permute_batched: the same stable counting sort as moe_permute (segment e holds the
 * slots with topk_idx == e in ascending flat index s = t*K + k; segment E the shared rows
 * of with_shared, ascending t), with the row of rank r in segment e at e*max_tokens + r.
 *   max_tokens >= 1; (E + with_shared) * max_tokens < 2^31.
 *   xb         [nseg * max_tokens, H]: BF16 copies, or E4M3 codes with xb_scales float32
 *              [nseg * max_tokens, H/128] (the 1x128 rule of moe_permute).
 *   masked_m   out int32 [nseg]: min(rows of segment e, max_tokens).
 *   src_row    out int32 [nseg * max_tokens]: source index of each real row, -1 elsewhere.
 *   inv_map    out int32 [T, K]: row of each slot; -1 for padding and for dropped slots.
 *   shared_map out int32 [T] (iff with_shared): the token's shared row, or -1.
 *   A segment with more than max_tokens rows keeps its first max_tokens (lowest flat
 *   index) and drops the rest: their inv_map / shared_map entries are -1 and
 *   MOE_DEV_OVERFLOW is ORed into dev_status.  (With distinct experts per token a segment
 *   holds at most T rows, so max_tokens >= T never drops.)
 *   ws         at least moe_permute_batched_workspace_bytes(T, K, E, with_shared) bytes.
 *   dispatch_scale, dispatch_format, topk_w, row_weights: as moe_permute_ex (row_weights
 *              [nseg*max_tokens]).
 * Errors: as moe_permute_ex. */
size_t moe_permute_batched_workspace_bytes(int T, int K, int E, int with_shared);
moe_status_t moe_permute_batched(const int32_t* topk_idx, int T, int K, int E, int with_shared,
                                 int max_tokens, const uint16_t* x, int H, moe_dtype_t out_dtype, void* xb,
                                 float* xb_scales, int32_t* masked_m, int32_t* src_row, int32_t* inv_map,
                                 int32_t* shared_map, void* ws, size_t ws_bytes, int32_t* dev_status,
                                 const float* dispatch_scale, int dispatch_format, const float* topk_w,
                                 float* row_weights, void* stream);

/* moe_grouped_gemm_ex over the batched layout: segment s covers rows
 * [s*max_tokens, s*max_tokens + min(max(masked_m[s], 0), max_tokens)) of a, out,
 * a_scales, out_scales and row_scale, all with nseg * max_tokens rows; masked_m is int32
 * [num_segments] on the device (read by the kernel: no host synchronisation).  Every other
 * argument, the arithmetic and the errors are those of moe_grouped_gemm_ex; rows past a
 * segment's masked_m are neither read into a result nor written. */
moe_status_t moe_grouped_gemm_batched(const void* a, const float* a_scales, const int32_t* masked_m,
                                      int num_segments, int max_tokens, int k_dim, int n_dim, const void* w,
                                      const float* w_scales, int num_w, const void* w_extra,
                                      const float* w_extra_scales, moe_dtype_t dtype, moe_epilogue_t epilogue,
                                      void* out, float* out_scales, int32_t* dev_status,
                                      const float* row_scale, void* stream);

/* ------------------------------------------------------- down projection + combine
 * The down projection with the combine fused into its epilogue ([MegaMoE]: one kernel
 * runs the expert GEMMs and the combine and leaves the weighted per-(token, slot) rows in
 * its buffer; here only the single-GPU part of that idea: no dispatch, no all-to-all).
 * It computes exactly what moe_grouped_gemm_ex (MOE_EPI_NONE) into y followed by
 * moe_combine(y, inv_map, topk_w, T, K, n_dim, y, shared_map, fq_scale, out) computes, bit for
 * bit, without the second launch and without reading y back from HBM: the warp whose
 * stores complete a token's rows in a 128-column block sums that block from L2 in the
 * combine's fixed order (a "last writer sums" scheme; the counts are atomic, the sums are
 * not, and no block ever waits for another).
 *   a ... dtype   as moe_grouped_gemm_ex; seg is cu_seqlens [num_segments + 1] when
 *              max_tokens == 0 (rows_cap rows), or masked_m [num_segments] of the batched
 *              layout when max_tokens > 0 (rows_cap is then num_segments * max_tokens).
 *   y          out BF16 [rows_cap, n_dim]: the expert rows (router-weighted if row_scale).
 *   src_row    int32 [rows_cap] from the permute (row -> t*K + k, or T*K + t for a shared row).
 *   inv_map, topk_w (nullable: rows already weighted), T, K, shared_map (nullable),
 *   fq_scale (nullable)   as moe_combine, with H = n_dim and y as the shared rows.
 *   out        BF16 [T, n_dim], every row written (+0 for a token with no row).
 *   counters   int32 [T, n_dim/128]: zero on entry; the call leaves it zero (after a
 *              MOE_DEV_PIPELINE_TIMEOUT the caller zeroes it again).
 * Errors: those of moe_grouped_gemm_ex; MOE_ERR_ARG for a null src_row / inv_map / out /
 * counters, or T > 0 with no row capacity. */
moe_status_t moe_grouped_gemm_combine(const void* a, const float* a_scales, const int32_t* seg,
                                      int num_segments, int max_tokens, int rows_cap, int k_dim, int n_dim,
                                      const void* w, const float* w_scales, int num_w, const void* w_extra,
                                      const float* w_extra_scales, moe_dtype_t dtype, uint16_t* y,
                                      const float* row_scale, const int32_t* src_row, const int32_t* inv_map,
                                      const float* topk_w, int T, int K, const int32_t* shared_map,
                                      const float* fq_scale, uint16_t* out, int32_t* counters,
                                      int32_t* dev_status, void* stream);

/* -------------------------------------------------------------------------- combine
 * Fixed-order combine ([MegaMoE]: each token's router-weighted slot rows are added in
 * increasing slot order into a float32 accumulator that starts at zero, rounded to BF16
 * a single time, with the fused shared expert added as the final, never-quantised slot):
 *     acc = +0.0f
 *     for k = 0..K-1 with inv_map[t,k] >= 0:
 *         r = float(y[inv_map[t,k]]) * topk_w[t,k]          (float32 product)
 *         if fq_scale: r = float(e4m3_rn_satfinite(r * s)) / s    (fake-quant, float32)
 *         acc = acc + r                                     (float32, no FMA)
 *     if the token has a valid slot and shared_y: acc = acc + float(shared row)
 *     out[t] = bf16_rn(acc)                   (a token with no valid slot gets +0)
 *   y          BF16 [rows, H] expert outputs in the permuted layout.
 *   inv_map    int32 [T, K] from moe_permute (-1 = padding slot, never read).
 *   topk_w     float32 [T, K]; NULL when the rows are already router-weighted (then
 *              r = float(y[...]), the same result as weights of 1).
 *   shared_y   nullable BF16: the shared expert's rows; row of token t is shared_map[t]
 *              when shared_map is given (e.g. y itself with moe_permute's shared_map),
 *              else t.
 *   fq_scale   nullable device float32 scalar s ([MegaMoE]: a calibrated or constant
 *              global combine scale; here s = 448 / amax).
 *   out        BF16 [T, H].
 * Bit-exact against a float32 reference given the same y rows. */
moe_status_t moe_combine(const uint16_t* y, const int32_t* inv_map, const float* topk_w, int T, int K,
                         int H, const uint16_t* shared_y, const int32_t* shared_map,
                         const float* fq_scale, uint16_t* out, void* stream);

/* Layout self-check ([MegaMoE]: on the first routed batch the re-summed rows must equal
 * the kernel's output exactly, and a captured graph performs that comparison on the
 * device).  Recomputes the
 * combine from the same arguments and compares it bit for bit with `expected`
 * (BF16 [T, H]); any difference ORs MOE_DEV_VERIFY_MISMATCH into dev_status (required).
 * Never asserts or traps. */
moe_status_t moe_combine_verify(const uint16_t* y, const int32_t* inv_map, const float* topk_w, int T,
                                int K, int H, const uint16_t* shared_y, const int32_t* shared_map,
                                const float* fq_scale, const uint16_t* expected, int32_t* dev_status,
                                void* stream);

/* Calibration ([MegaMoE]: max calibration, whose amax is the largest magnitude the
 * combine quantiser observes): amax = max(amax, max |float(y[inv_map[t,k]]) * topk_w[t,k]|) over
 * every valid slot.  amax is a device float32 the caller zeroes first; repeated calls
 * accumulate (max).  Exact (max is order-independent). */
moe_status_t moe_combine_amax(const uint16_t* y, const int32_t* inv_map, const float* topk_w, int T,
                              int K, int H, float* amax, void* stream);
/* scale = 448 / amax in float32 (1 if amax is 0), on the device. */
moe_status_t moe_fq_scale_from_amax(const float* amax, float* scale, void* stream);

/* Combine with NVFP4 fake-quant ([MegaMoE] runs its combine quantiser with NVFP4 units as
 * well as FP8 ones; the page leaves the format's arithmetic to that recipe, and this is the
 * two-level NVFP4 reading).  The same fixed-order sum as moe_combine, with every
 * router-weighted routed row r fake-quantised per block of 16 consecutive columns, in
 * float32 with IEEE roundings:
 *     a = max |r| over the block
 *     s_b = e4m3(fl32(fl32(a / 6) * g))          (nearest even, saturating; E4M3 block scale)
 *     inv = fl32(g / s_b)  (0 if s_b is 0);  d = fl32(s_b / g)
 *     r' = fl32(e2m1(fl32(r * inv)) * d)          (E2M1: 0, .5, 1, 1.5, 2, 3, 4, 6; nearest
 *                                                  even, saturating at 6; sign kept)
 * The shared slot is added last and unquantised.
 *   g_scale    device float32: the per-tensor scale g (moe_fq4_scale_from_amax).
 *   Other arguments and errors as moe_combine (H a multiple of 128, so of 16). */
moe_status_t moe_combine_nvfp4(const uint16_t* y, const int32_t* inv_map, const float* topk_w, int T, int K,
                               int H, const uint16_t* shared_y, const int32_t* shared_map,
                               const float* g_scale, uint16_t* out, void* stream);
/* NVFP4 per-tensor scale g = 448 * 6 / amax in float32 (1 if amax is 0), on the device:
 * the largest block (amax / 6) maps onto the largest E4M3 block scale.  amax as from
 * moe_combine_amax. */
moe_status_t moe_fq4_scale_from_amax(const float* amax, float* scale, void* stream);

/* ---------------------------------------------------------------------------- layer
 * The whole layer in one call, one stream, no host synchronisation:
 *   route (if logits) -> permute (+ FP8 quantisation for E4M3) -> grouped GEMM gate/up
 *   with fused SwiGLU -> grouped GEMM down -> combine.  The shared expert, when present,
 *   is segment E of both grouped GEMMs (it must have the routed experts' I). */
typedef struct {
  int T;              /* rows of the batch (a receive bucket may pad them) */
  int H, I, E, K;
  moe_dtype_t dtype;  /* MOE_BF16, or MOE_E4M3 (weights and activations FP8, 128-blocks) */
  int has_shared;     /* 1: one shared expert, added last in the combine, never quantised */
  int weight_in_down; /* 1: router weights applied in the down projection's epilogue (rows
                         stored weighted in BF16, the combine only sums); 0: in the combine */
  int max_tokens;     /* 0: contiguous expert-major layout (cu_seqlens); > 0: the batched
                         layout, max_tokens rows per segment (the shared expert's included),
                         through moe_permute_batched / moe_grouped_gemm_batched (ABI 3) */
  int fuse_combine;   /* 1: the combine runs inside the down projection
                         (moe_grouped_gemm_combine); same output bit for bit (ABI 3) */
  int combine_fq_format; /* with a combine fake-quant scale: 0 E4M3 (moe_combine), 1 NVFP4
                            (moe_combine_nvfp4; not with fuse_combine) (ABI 4) */
  int dispatch_fq_format; /* with a dispatch fake-quant scale: 0 E4M3, 1 NVFP4 (ABI 4) */
  int gemm_pairs;     /* 1: both grouped GEMMs on SM pairs (moe_grouped_gemm_pairs; BF16,
                         contiguous layout, not with fuse_combine, else MOE_ERR_UNSUPPORTED);
                         same output bit for bit; 0: moe_grouped_gemm / _ex (ABI 5) */
  int weight_tiles;   /* 1: w13, w2, shared_w13 and shared_w2 are in the tile layout of
                         moe_pack_weights (any layout and dtype; not with gemm_pairs, else
                         MOE_ERR_UNSUPPORTED); same output bit for bit; 0: row-major (ABI 6) */
} moe_layer_desc_t;

typedef struct {
  const void* w13;        /* [E, 2I, H] gate rows then up rows, BF16 or E4M3 */
  const float* w13_scales;/* E4M3 only: [E, 2I/128, H/128] */
  const void* w2;         /* [E, H, I] */
  const float* w2_scales; /* E4M3 only: [E, H/128, I/128] */
  const void* shared_w13; /* has_shared: [2I, H] */
  const float* shared_w13_scales;
  const void* shared_w2;  /* has_shared: [H, I] */
  const float* shared_w2_scales;
} moe_layer_weights_t;

/* Pointers into a layer workspace, for inspection and calibration (all device). */
typedef struct {
  void* xp; float* xp_scales;   /* permuted activations [cap, H] (+ [cap, H/128]) */
  void* hs; float* hs_scales;   /* SwiGLU output [cap, I] (+ [cap, I/128]) */
  uint16_t* y;                  /* expert outputs BF16 [cap, H] */
  int32_t* cu_seqlens;          /* [E + has_shared + 1] */
  int32_t* src_row;             /* [cap] */
  int32_t* inv_map;             /* [T, K] */
  int32_t* shared_map;          /* [T] or NULL */
  float* row_weights;           /* [cap] router weight per row (weight_in_down) */
  int cap;                      /* T*K + (has_shared ? T : 0); batched: nseg * max_tokens */
  int32_t* masked_m;            /* batched layout: [E + has_shared] rows per segment; else NULL
                                   (and cu_seqlens is NULL in the batched layout) */
  int32_t* counters;            /* fuse_combine: [T, H/128] (zeroed by the layer's permute); else NULL */
} moe_layer_views_t;

/* Workspace bytes for a layer of this shape (0 for an invalid descriptor). */
size_t moe_layer_workspace_bytes(const moe_layer_desc_t* d);
/* Fill `views` (host struct) with the sub-buffers of `ws`. */
moe_status_t moe_layer_views(const moe_layer_desc_t* d, void* ws, moe_layer_views_t* views);

/*   d, w       host structs (read during the call only).
 *   logits     nullable float32 [T, E]: route inside the layer (num_tokens as in
 *              moe_route_topk) and write topk_idx / topk_w; NULL: topk_idx / topk_w are
 *              inputs (e.g. routed elsewhere, with padding slots set to -1 by the caller).
 *   x          BF16 [T, H];  fq_scale nullable device scalar (combine fake-quant: the
 *              E4M3 scale, or the NVFP4 per-tensor scale when d->combine_fq_format is 1);
 *   dispatch_scale nullable device scalar (dispatch fake-quant, BF16 layers; see
 *              moe_permute_ex);
 *   out        BF16 [T, H];  ws / ws_bytes: workspace, 256-byte aligned.
 * Errors: as the step calls; MOE_ERR_WORKSPACE if ws_bytes < moe_layer_workspace_bytes;
 * MOE_ERR_UNSUPPORTED for an NVFP4 combine fake-quant with fuse_combine. */
moe_status_t moe_layer_forward(const moe_layer_desc_t* d, const moe_layer_weights_t* w,
                               const float* logits, const int32_t* num_tokens, int32_t* topk_idx,
                               float* topk_w, const uint16_t* x, const float* fq_scale,
                               const float* dispatch_scale, uint16_t* out, void* ws, size_t ws_bytes,
                               int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
