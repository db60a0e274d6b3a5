// The whole MoE layer on one stream with no host synchronisation (so it can be captured
// in a CUDA graph, the constraint the Mega-MoE page puts on its combine after the first
// check): route -> permute (+FP8 quantisation) -> grouped GEMM gate/up with fused SwiGLU
// -> grouped GEMM down -> fixed-order combine.  The shared expert is segment E of both
// grouped GEMMs and the last slot of the combine.
//
// Workspace (caller-owned, sized from the layer's actual shape -- the permute-scratch
// page's rule -- every region 256-byte aligned):
//   cu_seqlens [E+2] | src_row [cap] | inv_map [T*K] | shared_map [T] | permute scratch |
//   xp [cap, H] (+ scales [cap, H/128]) | hs [cap, I] (+ scales [cap, I/128]) | y [cap, H] bf16
// with cap = T*K + (has_shared ? T : 0).  The batched layout (max_tokens > 0) has
// cap = (E + has_shared) * max_tokens rows, masked_m [E+1] in place of cu_seqlens, and the
// batched permute's scratch (which keeps its cu_seqlens internal).
#include "common.cuh"

namespace moe {

struct LayerPlan {
  size_t off_cu, off_src, off_inv, off_smap, off_roww, off_scratch, off_xp, off_xps, off_hs, off_hss, off_y, off_cnt,
      total;
  size_t scratch_bytes;
  int cap, nseg;
};

inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

inline bool plan_layer(const moe_layer_desc_t* d, LayerPlan* p) {
  if (!d) return false;
  if (d->T < 0 || d->H <= 0 || d->I <= 0 || d->E < 1 || d->E > kMaxExperts || d->K < 1 || d->K > d->E ||
      d->K > kMaxTopK || d->H % 128 || d->I % 128 || (d->has_shared != 0 && d->has_shared != 1) ||
      (d->weight_in_down != 0 && d->weight_in_down != 1) || d->max_tokens < 0 ||
      (d->fuse_combine != 0 && d->fuse_combine != 1) ||
      (d->combine_fq_format != 0 && d->combine_fq_format != 1) ||
      (d->dispatch_fq_format != 0 && d->dispatch_fq_format != 1) ||
      (d->gemm_pairs != 0 && d->gemm_pairs != 1) || (d->weight_tiles != 0 && d->weight_tiles != 1) ||
      (d->dtype != MOE_BF16 && d->dtype != MOE_E4M3))
    return false;
  const size_t T = d->T, K = d->K, H = d->H, I = d->I;
  const bool batched = d->max_tokens > 0;
  const size_t nseg = (size_t)d->E + d->has_shared;
  const size_t cap = batched ? nseg * (size_t)d->max_tokens : T * K + (d->has_shared ? T : 0);
  if (cap > 0x7fffffffull || T * K + T > 0x7fffffffull) return false;
  const size_t esz = d->dtype == MOE_E4M3 ? 1 : 2;
  const bool fp8 = d->dtype == MOE_E4M3;
  p->cap = (int)cap;
  p->nseg = (int)nseg;
  p->scratch_bytes = batched ? moe_permute_batched_workspace_bytes(d->T, d->K, d->E, d->has_shared)
                             : moe_permute_workspace_bytes(d->T, d->K, d->E, d->has_shared);
  size_t o = 0;
  p->off_cu = o;      o = align256(o + 4 * (size_t)(p->nseg + 1));
  p->off_src = o;     o = align256(o + 4 * cap);
  p->off_inv = o;     o = align256(o + 4 * T * K);
  p->off_smap = o;    o = align256(o + 4 * T);
  p->off_roww = o;    o = align256(o + 4 * cap);
  p->off_scratch = o; o = align256(o + p->scratch_bytes);
  p->off_xp = o;      o = align256(o + cap * H * esz);
  p->off_xps = o;     o = align256(o + (fp8 ? cap * (H / 128) * 4 : 0));
  p->off_hs = o;      o = align256(o + cap * I * esz);
  p->off_hss = o;     o = align256(o + (fp8 ? cap * (I / 128) * 4 : 0));
  p->off_y = o;       o = align256(o + cap * H * 2);
  p->off_cnt = o;     o = align256(o + (d->fuse_combine ? T * (H / 128) * 4 : 0));
  p->total = o;
  return true;
}

}  // namespace moe

extern "C" size_t moe_layer_workspace_bytes(const moe_layer_desc_t* d) {
  moe::LayerPlan p;
  return moe::plan_layer(d, &p) ? p.total : 0;
}

extern "C" moe_status_t moe_layer_views(const moe_layer_desc_t* d, void* ws, moe_layer_views_t* v) {
  moe::LayerPlan p;
  if (!moe::plan_layer(d, &p) || !ws || !v) return MOE_ERR_ARG;
  uint8_t* b = static_cast<uint8_t*>(ws);
  const bool fp8 = d->dtype == MOE_E4M3;
  const bool batched = d->max_tokens > 0;
  // one region: cu_seqlens [nseg + 1] in the contiguous layout, masked_m [nseg] in the batched
  v->cu_seqlens = batched ? nullptr : reinterpret_cast<int32_t*>(b + p.off_cu);
  v->masked_m = batched ? reinterpret_cast<int32_t*>(b + p.off_cu) : nullptr;
  v->src_row = reinterpret_cast<int32_t*>(b + p.off_src);
  v->inv_map = reinterpret_cast<int32_t*>(b + p.off_inv);
  v->shared_map = d->has_shared ? reinterpret_cast<int32_t*>(b + p.off_smap) : nullptr;
  v->row_weights = reinterpret_cast<float*>(b + p.off_roww);
  v->xp = b + p.off_xp;
  v->xp_scales = fp8 ? reinterpret_cast<float*>(b + p.off_xps) : nullptr;
  v->hs = b + p.off_hs;
  v->hs_scales = fp8 ? reinterpret_cast<float*>(b + p.off_hss) : nullptr;
  v->y = reinterpret_cast<uint16_t*>(b + p.off_y);
  v->counters = d->fuse_combine ? reinterpret_cast<int32_t*>(b + p.off_cnt) : nullptr;
  v->cap = p.cap;
  return MOE_OK;
}

extern "C" moe_status_t moe_layer_forward(const moe_layer_desc_t* d, const moe_layer_weights_t* w,
                                          const float* logits, const int32_t* num_tokens, int32_t* topk_idx,
                                          float* topk_w, const uint16_t* x, const float* fq_scale,
                                          const float* dispatch_scale, uint16_t* out, void* ws, size_t ws_bytes,
                                          int32_t* dev_status, void* stream) {
  using namespace moe;
  LayerPlan p;
  if (!plan_layer(d, &p) || !w) return MOE_ERR_ARG;
  if (!ws || ws_bytes < p.total) return MOE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255) return MOE_ERR_ARG;
  if (d->T == 0) return MOE_OK;
  if (!topk_idx || !topk_w || !x || !out || !w->w13 || !w->w2) return MOE_ERR_ARG;
  const bool fp8 = d->dtype == MOE_E4M3;
  if (fp8 && (!w->w13_scales || !w->w2_scales)) return MOE_ERR_ARG;
  if (fp8 && dispatch_scale) return MOE_ERR_UNSUPPORTED;   // the FP8 path already quantises the dispatch
  const bool fq4 = fq_scale && d->combine_fq_format == 1;
  if (fq4 && d->fuse_combine) return MOE_ERR_UNSUPPORTED;
  if (d->gemm_pairs && (fp8 || d->max_tokens > 0 || d->fuse_combine || d->weight_tiles)) return MOE_ERR_UNSUPPORTED;
  if (d->has_shared && (!w->shared_w13 || !w->shared_w2 ||
                        (fp8 && (!w->shared_w13_scales || !w->shared_w2_scales))))
    return MOE_ERR_ARG;
  moe_layer_views_t v;
  moe_layer_views(d, ws, &v);
  moe_status_t st;
  if (logits) {
    st = moe_route_topk(logits, d->T, d->E, d->K, num_tokens, topk_idx, topk_w, stream);
    if (st != MOE_OK) return st;
  }
  const bool wd = d->weight_in_down != 0;
  const void* sx13 = d->has_shared ? w->shared_w13 : nullptr;
  const void* sx2 = d->has_shared ? w->shared_w2 : nullptr;
  const float* sx13s = d->has_shared ? w->shared_w13_scales : nullptr;
  const float* sx2s = d->has_shared ? w->shared_w2_scales : nullptr;
  // the grouped GEMMs' dtype argument, with the weight layout
  const moe_dtype_t gdt = static_cast<moe_dtype_t>(d->dtype | (d->weight_tiles ? MOE_W_TILED : 0));
  if (d->max_tokens > 0) {
    // batched layout: same steps, segment s in rows [s*max_tokens, s*max_tokens + masked_m[s])
    const int mt = d->max_tokens;
    if (mt < 1) return MOE_ERR_ARG;
    st = permute_impl(topk_idx, d->T, d->K, d->E, d->has_shared, x, d->H, d->dtype, v.xp, v.xp_scales, nullptr,
                      v.src_row, v.inv_map, v.shared_map, static_cast<uint8_t*>(ws) + p.off_scratch,
                      p.scratch_bytes, dev_status, dispatch_scale, wd ? topk_w : nullptr,
                      wd ? v.row_weights : nullptr, mt, v.masked_m, stream, v.counters, d->H / 128,
                      d->dispatch_fq_format);
    if (st != MOE_OK) return st;
    st = moe_grouped_gemm_batched(v.xp, v.xp_scales, v.masked_m, p.nseg, mt, d->H, 2 * d->I, w->w13,
                                  w->w13_scales, d->E, sx13, sx13s, gdt, MOE_EPI_SWIGLU, v.hs, v.hs_scales,
                                  dev_status, nullptr, stream);
    if (st != MOE_OK) return st;
    if (d->fuse_combine)
      return moe_grouped_gemm_combine(v.hs, v.hs_scales, v.masked_m, p.nseg, mt, 0, d->I, d->H, w->w2,
                                      w->w2_scales, d->E, sx2, sx2s, gdt, v.y, wd ? v.row_weights : nullptr,
                                      v.src_row, v.inv_map, wd ? nullptr : topk_w, d->T, d->K, v.shared_map,
                                      fq_scale, out, v.counters, dev_status, stream);
    st = moe_grouped_gemm_batched(v.hs, v.hs_scales, v.masked_m, p.nseg, mt, d->I, d->H, w->w2, w->w2_scales,
                                  d->E, sx2, sx2s, gdt, MOE_EPI_NONE, v.y, nullptr, dev_status,
                                  wd ? v.row_weights : nullptr, stream);
    if (st != MOE_OK) return st;
    if (fq4)
      return moe_combine_nvfp4(v.y, v.inv_map, wd ? nullptr : topk_w, d->T, d->K, d->H,
                               d->has_shared ? v.y : nullptr, v.shared_map, fq_scale, out, stream);
    return moe_combine(v.y, v.inv_map, wd ? nullptr : topk_w, d->T, d->K, d->H, d->has_shared ? v.y : nullptr,
                       v.shared_map, fq_scale, out, stream);
  }
  st = permute_impl(topk_idx, d->T, d->K, d->E, d->has_shared, x, d->H, d->dtype, v.xp, v.xp_scales, v.cu_seqlens,
                    v.src_row, v.inv_map, v.shared_map, static_cast<uint8_t*>(ws) + p.off_scratch, p.scratch_bytes,
                    dev_status, dispatch_scale, wd ? topk_w : nullptr, wd ? v.row_weights : nullptr, 0, nullptr,
                    stream, v.counters, d->H / 128, d->dispatch_fq_format);
  if (st != MOE_OK) return st;
  if (d->gemm_pairs) {
    st = moe_grouped_gemm_pairs(v.xp, v.cu_seqlens, p.nseg, p.cap, d->H, 2 * d->I, w->w13, d->E, sx13, MOE_EPI_SWIGLU,
                                v.hs, dev_status, nullptr, stream);
    if (st != MOE_OK) return st;
    st = moe_grouped_gemm_pairs(v.hs, v.cu_seqlens, p.nseg, p.cap, d->I, d->H, w->w2, d->E, sx2, MOE_EPI_NONE, v.y,
                                dev_status, wd ? v.row_weights : nullptr, stream);
    if (st != MOE_OK) return st;
    if (fq4)
      return moe_combine_nvfp4(v.y, v.inv_map, wd ? nullptr : topk_w, d->T, d->K, d->H,
                               d->has_shared ? v.y : nullptr, v.shared_map, fq_scale, out, stream);
    return moe_combine(v.y, v.inv_map, wd ? nullptr : topk_w, d->T, d->K, d->H, d->has_shared ? v.y : nullptr,
                       v.shared_map, fq_scale, out, stream);
  }
  st = moe_grouped_gemm(v.xp, v.xp_scales, v.cu_seqlens, p.nseg, p.cap, d->H, 2 * d->I, w->w13, w->w13_scales, d->E,
                        sx13, d->has_shared ? w->shared_w13_scales : nullptr, gdt, MOE_EPI_SWIGLU, v.hs,
                        v.hs_scales, dev_status, stream);
  if (st != MOE_OK) return st;
  if (d->fuse_combine)
    return moe_grouped_gemm_combine(v.hs, v.hs_scales, v.cu_seqlens, p.nseg, 0, p.cap, d->I, d->H, w->w2,
                                    w->w2_scales, d->E, sx2, sx2s, gdt, v.y, wd ? v.row_weights : nullptr,
                                    v.src_row, v.inv_map, wd ? nullptr : topk_w, d->T, d->K, v.shared_map, fq_scale,
                                    out, v.counters, dev_status, stream);
  st = moe_grouped_gemm_ex(v.hs, v.hs_scales, v.cu_seqlens, p.nseg, p.cap, d->I, d->H, w->w2, w->w2_scales, d->E,
                           sx2, d->has_shared ? w->shared_w2_scales : nullptr, gdt, MOE_EPI_NONE, v.y, nullptr,
                           dev_status, wd ? v.row_weights : nullptr, stream);
  if (st != MOE_OK) return st;
  // with the router weights applied in the down projection the combine only sums
  if (fq4)
    return moe_combine_nvfp4(v.y, v.inv_map, wd ? nullptr : topk_w, d->T, d->K, d->H,
                             d->has_shared ? v.y : nullptr, v.shared_map, fq_scale, out, stream);
  return moe_combine(v.y, v.inv_map, wd ? nullptr : topk_w, d->T, d->K, d->H, d->has_shared ? v.y : nullptr,
                     v.shared_map, fq_scale, out, stream);
}
