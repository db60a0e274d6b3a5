"""Python binding of libmoe (include/moe.h): argument marshalling only.

Every function has the name of the C entry point it calls and forwards torch tensors as
raw device pointers plus sizes; every step of the layer runs in the library's own CUDA
kernels.  PyTorch is used for device memory and streams only.  If libmoe.so has not been
built, the first call raises: there is no CPU or PyTorch fallback.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_BF16, MOE_E4M3 = 0, 1
MOE_W_TILED = 0x100   # ORed into a grouped GEMM dtype: weights in the tile layout of moe_pack_weights
MOE_EPI_NONE, MOE_EPI_SWIGLU = 0, 1
MOE_DEV_BAD_EXPERT, MOE_DEV_VERIFY_MISMATCH, MOE_DEV_PIPELINE_TIMEOUT, MOE_DEV_OVERFLOW = 1, 2, 4, 8
STATUS = {0: "MOE_OK", 1: "MOE_ERR_ARG", 2: "MOE_ERR_WORKSPACE", 3: "MOE_ERR_UNSUPPORTED", 4: "MOE_ERR_CUDA"}

_P, _I, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t


class MoeError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


class LayerDesc(ctypes.Structure):
    _fields_ = [("T", _I), ("H", _I), ("I", _I), ("E", _I), ("K", _I), ("dtype", _I), ("has_shared", _I),
                ("weight_in_down", _I), ("max_tokens", _I), ("fuse_combine", _I), ("combine_fq_format", _I),
                ("dispatch_fq_format", _I), ("gemm_pairs", _I), ("weight_tiles", _I)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("w13", "w13_scales", "w2", "w2_scales", "shared_w13", "shared_w13_scales",
                                  "shared_w2", "shared_w2_scales")]


class LayerViews(ctypes.Structure):
    _fields_ = [("xp", _P), ("xp_scales", _P), ("hs", _P), ("hs_scales", _P), ("y", _P), ("cu_seqlens", _P),
                ("src_row", _P), ("inv_map", _P), ("shared_map", _P), ("row_weights", _P), ("cap", _I),
                ("masked_m", _P), ("counters", _P)]


# C signatures (restype int = moe_status_t unless noted)
_SIGS = {
    "moe_abi_version": ([], _I),
    "moe_status_string": ([_I], ctypes.c_char_p),
    "moe_route_topk": ([_P, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_permute_workspace_bytes": ([_I, _I, _I, _I], _Z),
    "moe_permute": ([_P, _I, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _Z, _P, _P], _I),
    "moe_permute_noalloc_max_scratch_bytes": ([], _Z),
    "moe_permute_noalloc": ([_P, _I, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_permute_ex": ([_P, _I, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _Z, _P, _P, _I, _P, _P, _P], _I),
    "moe_permute_batched_workspace_bytes": ([_I, _I, _I, _I], _Z),
    "moe_permute_batched": ([_P, _I, _I, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _Z, _P, _P, _I, _P,
                             _P, _P], _I),
    "moe_amax_bf16": ([_P, _Z, _P, _P], _I),
    "moe_quantize_act_fp8": ([_P, _I, _I, _P, _P, _P], _I),
    "moe_quantize_weight_fp8": ([_P, _I, _I, _I, _P, _P, _P], _I),
    "moe_grouped_gemm": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P, _I, _I, _P, _P, _P, _P], _I),
    "moe_grouped_gemm_ex": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P, _I, _I, _P, _P, _P, _P, _P], _I),
    "moe_grouped_gemm_pairs": ([_P, _P, _I, _I, _I, _I, _P, _I, _P, _I, _P, _P, _P, _P], _I),
    "moe_pack_weights": ([_P, _I, _I, _I, _I, _P, _P], _I),
    "moe_grouped_gemm_batched": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P, _I, _I, _P, _P, _P, _P, _P],
                                 _I),
    "moe_grouped_gemm_combine": ([_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P, _I, _P, _P, _P, _P, _P, _I,
                                  _I, _P, _P, _P, _P, _P, _P], _I),
    "moe_combine": ([_P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "moe_combine_verify": ([_P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P], _I),
    "moe_combine_amax": ([_P, _P, _P, _I, _I, _I, _P, _P], _I),
    "moe_fq_scale_from_amax": ([_P, _P, _P], _I),
    "moe_combine_nvfp4": ([_P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "moe_fq4_scale_from_amax": ([_P, _P, _P], _I),
    "moe_layer_workspace_bytes": ([ctypes.POINTER(LayerDesc)], _Z),
    "moe_layer_views": ([ctypes.POINTER(LayerDesc), _P, ctypes.POINTER(LayerViews)], _I),
    "moe_layer_forward": ([ctypes.POINTER(LayerDesc), ctypes.POINTER(LayerWeights), _P, _P, _P, _P, _P, _P, _P,
                           _P, _P, _Z, _P, _P], _I),
}

_lib = None


def lib():
    """The loaded libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m combine_moe_route_softmax_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn, code):
    if code != 0:
        raise MoeError(fn, code)


def _dev(t):
    assert t.is_cuda and t.is_contiguous(), "expected a contiguous CUDA tensor"
    return t


# ----------------------------------------------------------------------------- calls
def moe_route_topk(logits, K, num_tokens=None, topk_idx=None, topk_w=None, stream=None):
    _dev(logits)
    T, E = logits.shape
    if topk_idx is None:
        topk_idx = torch.empty(T, K, dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty(T, K, dtype=torch.float32, device=logits.device)
    _check("moe_route_topk", lib().moe_route_topk(_ptr(logits), T, E, K, _ptr(num_tokens), _ptr(topk_idx),
                                                  _ptr(topk_w), _stream(stream)))
    return topk_idx, topk_w


def moe_permute_workspace_bytes(T, K, E, with_shared):
    return lib().moe_permute_workspace_bytes(T, K, E, int(with_shared))


def _fmt(name):
    """Fake-quant format name -> the C code (0 E4M3, 1 NVFP4)."""
    if name not in ("e4m3", "nvfp4"):
        raise ValueError("fake-quant format is 'e4m3' or 'nvfp4'")
    return int(name == "nvfp4")


def moe_permute(topk_idx, E, x, with_shared=False, out_dtype=MOE_BF16, ws=None, dev_status=None, stream=None,
                dispatch_scale=None, topk_w=None, dispatch_format="e4m3"):
    """Returns dict(xp, xp_scales, cu_seqlens, src_row, inv_map, shared_map, row_weights).
    dispatch_scale / topk_w select moe_permute_ex (dispatch fake-quant in dispatch_format
    "e4m3" or "nvfp4" / row weights)."""
    _dev(topk_idx)
    _dev(x)
    T, K = topk_idx.shape
    H = x.shape[1]
    dev = x.device
    cap = T * K + (T if with_shared else 0)
    nseg = E + int(with_shared)
    fp8 = out_dtype == MOE_E4M3
    xp = torch.empty(cap, H, dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    xps = torch.empty(cap, H // 128, dtype=torch.float32, device=dev) if fp8 else None
    cu = torch.empty(nseg + 1, dtype=torch.int32, device=dev)
    src = torch.empty(cap, dtype=torch.int32, device=dev)
    inv = torch.empty(T, K, dtype=torch.int32, device=dev)
    smap = torch.empty(T, dtype=torch.int32, device=dev) if with_shared else None
    nbytes = moe_permute_workspace_bytes(T, K, E, with_shared)
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    roww = None
    if dispatch_scale is None and topk_w is None:
        _check("moe_permute", lib().moe_permute(
            _ptr(topk_idx), T, K, E, int(with_shared), _ptr(x), H, out_dtype, _ptr(xp), _ptr(xps), _ptr(cu),
            _ptr(src), _ptr(inv), _ptr(smap), _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status),
            _stream(stream)))
    else:
        if topk_w is not None:
            roww = torch.empty(cap, dtype=torch.float32, device=dev)
        _check("moe_permute_ex", lib().moe_permute_ex(
            _ptr(topk_idx), T, K, E, int(with_shared), _ptr(x), H, out_dtype, _ptr(xp), _ptr(xps), _ptr(cu),
            _ptr(src), _ptr(inv), _ptr(smap), _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status),
            _ptr(dispatch_scale), _fmt(dispatch_format), _ptr(topk_w), _ptr(roww), _stream(stream)))
    return dict(xp=xp, xp_scales=xps, cu_seqlens=cu, src_row=src, inv_map=inv, shared_map=smap, row_weights=roww)


def moe_permute_batched_workspace_bytes(T, K, E, with_shared):
    return lib().moe_permute_batched_workspace_bytes(T, K, E, int(with_shared))


def moe_permute_batched(topk_idx, E, x, max_tokens, with_shared=False, out_dtype=MOE_BF16, ws=None,
                        dev_status=None, stream=None, dispatch_scale=None, topk_w=None, dispatch_format="e4m3"):
    """Batched layout: returns dict(xb [nseg, max_tokens, H], xb_scales, masked_m [nseg], src_row
    [nseg * max_tokens], inv_map, shared_map, row_weights)."""
    _dev(topk_idx)
    _dev(x)
    T, K = topk_idx.shape
    H = x.shape[1]
    dev = x.device
    nseg = E + int(with_shared)
    rows = nseg * max_tokens
    fp8 = out_dtype == MOE_E4M3
    xb = torch.empty(nseg, max_tokens, H, dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    xbs = torch.empty(nseg, max_tokens, H // 128, dtype=torch.float32, device=dev) if fp8 else None
    mm = torch.empty(nseg, dtype=torch.int32, device=dev)
    src = torch.empty(rows, dtype=torch.int32, device=dev)
    inv = torch.empty(T, K, dtype=torch.int32, device=dev)
    smap = torch.empty(T, dtype=torch.int32, device=dev) if with_shared else None
    roww = torch.empty(rows, dtype=torch.float32, device=dev) if topk_w is not None else None
    if ws is None:
        ws = torch.empty(moe_permute_batched_workspace_bytes(T, K, E, with_shared), dtype=torch.uint8, device=dev)
    _check("moe_permute_batched", lib().moe_permute_batched(
        _ptr(topk_idx), T, K, E, int(with_shared), max_tokens, _ptr(x), H, out_dtype, _ptr(xb), _ptr(xbs), _ptr(mm),
        _ptr(src), _ptr(inv), _ptr(smap), _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status),
        _ptr(dispatch_scale), _fmt(dispatch_format), _ptr(topk_w), _ptr(roww), _stream(stream)))
    return dict(xb=xb, xb_scales=xbs, masked_m=mm, src_row=src, inv_map=inv, shared_map=smap, row_weights=roww)


def moe_quantize_act_fp8(x, stream=None):
    _dev(x)
    R, C = x.shape
    q = torch.empty(R, C, dtype=torch.uint8, device=x.device)
    s = torch.empty(R, C // 128, dtype=torch.float32, device=x.device)
    _check("moe_quantize_act_fp8", lib().moe_quantize_act_fp8(_ptr(x), R, C, _ptr(q), _ptr(s), _stream(stream)))
    return q, s


def moe_quantize_weight_fp8(w, stream=None):
    """w BF16 [..., rows, cols] -> (codes uint8 same shape, scales float32 [..., rows/128, cols/128])."""
    _dev(w)
    rows, cols = w.shape[-2:]
    mats = w.numel() // (rows * cols)
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    s = torch.empty(*w.shape[:-2], rows // 128, cols // 128, dtype=torch.float32, device=w.device)
    _check("moe_quantize_weight_fp8", lib().moe_quantize_weight_fp8(_ptr(w), mats, rows, cols, _ptr(q), _ptr(s),
                                                                    _stream(stream)))
    return q, s


def moe_pack_weights(w, out=None, stream=None):
    """w [..., n, k] (bf16, or uint8 E4M3 codes) -> a tensor of the same shape and dtype
    holding the same bytes in the tile layout of moe_pack_weights (pass it with tiled=True
    or to MoeLayer(weight_tiles=True) only: its rows are not w's rows)."""
    _dev(w)
    n, k = w.shape[-2:]
    mats = w.numel() // (n * k)
    if out is None:
        out = torch.empty_like(w)
    _dev(out)
    assert out.numel() * out.element_size() == w.numel() * w.element_size(), "out must hold w's bytes"
    dt = MOE_E4M3 if w.dtype == torch.uint8 else MOE_BF16
    _check("moe_pack_weights", lib().moe_pack_weights(_ptr(w), mats, n, k, dt, _ptr(out), _stream(stream)))
    return out


def moe_grouped_gemm(a, cu_seqlens, w, n_segments=None, a_scales=None, w_scales=None, w_extra=None,
                     w_extra_scales=None, epilogue=MOE_EPI_NONE, out=None, out_scales=None, dev_status=None,
                     stream=None, row_scale=None, pairs=False, tiled=False):
    """a [rows_cap, k] (bf16 or uint8 E4M3 codes); w [num_w, n, k]; returns (out, out_scales).
    pairs=True: the BF16 computation on pairs of SMs (moe_grouped_gemm_pairs); tiled=True: w
    and w_extra from moe_pack_weights (MOE_W_TILED)."""
    _dev(a)
    fp8 = a.dtype == torch.uint8
    rows_cap, k_dim = a.shape
    num_w, n_dim = w.shape[0], w.shape[1]
    if n_segments is None:
        n_segments = cu_seqlens.numel() - 1
    out_cols = n_dim // 2 if epilogue == MOE_EPI_SWIGLU else n_dim
    if out is None:
        odt = torch.uint8 if (fp8 and epilogue == MOE_EPI_SWIGLU) else torch.bfloat16
        out = torch.empty(rows_cap, out_cols, dtype=odt, device=a.device)
    if fp8 and epilogue == MOE_EPI_SWIGLU and out_scales is None:
        out_scales = torch.empty(rows_cap, out_cols // 128, dtype=torch.float32, device=a.device)
    dt = (MOE_E4M3 if fp8 else MOE_BF16) | (MOE_W_TILED if tiled else 0)
    if pairs:
        _check("moe_grouped_gemm_pairs", lib().moe_grouped_gemm_pairs(
            _ptr(a), _ptr(cu_seqlens), n_segments, rows_cap, k_dim, n_dim, _ptr(w), num_w, _ptr(w_extra), epilogue,
            _ptr(out), _ptr(dev_status), _ptr(row_scale), _stream(stream)))
    elif row_scale is None:
        _check("moe_grouped_gemm", lib().moe_grouped_gemm(
            _ptr(a), _ptr(a_scales), _ptr(cu_seqlens), n_segments, rows_cap, k_dim, n_dim, _ptr(w), _ptr(w_scales),
            num_w, _ptr(w_extra), _ptr(w_extra_scales), dt, epilogue, _ptr(out),
            _ptr(out_scales), _ptr(dev_status), _stream(stream)))
    else:
        _check("moe_grouped_gemm_ex", lib().moe_grouped_gemm_ex(
            _ptr(a), _ptr(a_scales), _ptr(cu_seqlens), n_segments, rows_cap, k_dim, n_dim, _ptr(w), _ptr(w_scales),
            num_w, _ptr(w_extra), _ptr(w_extra_scales), dt, epilogue, _ptr(out),
            _ptr(out_scales), _ptr(dev_status), _ptr(row_scale), _stream(stream)))
    return out, out_scales


def moe_grouped_gemm_batched(a, masked_m, w, a_scales=None, w_scales=None, w_extra=None, w_extra_scales=None,
                             epilogue=MOE_EPI_NONE, out=None, out_scales=None, dev_status=None, stream=None,
                             row_scale=None, tiled=False):
    """a [S, max_tokens, k] (bf16 or uint8 E4M3 codes), masked_m int32 [S]; w [num_w, n, k];
    returns (out [S, max_tokens, n_out], out_scales)."""
    _dev(a)
    fp8 = a.dtype == torch.uint8
    S, max_tokens, k_dim = a.shape
    num_w, n_dim = w.shape[0], w.shape[1]
    out_cols = n_dim // 2 if epilogue == MOE_EPI_SWIGLU else n_dim
    if out is None:
        odt = torch.uint8 if (fp8 and epilogue == MOE_EPI_SWIGLU) else torch.bfloat16
        out = torch.empty(S, max_tokens, out_cols, dtype=odt, device=a.device)
    if fp8 and epilogue == MOE_EPI_SWIGLU and out_scales is None:
        out_scales = torch.empty(S, max_tokens, out_cols // 128, dtype=torch.float32, device=a.device)
    _check("moe_grouped_gemm_batched", lib().moe_grouped_gemm_batched(
        _ptr(a), _ptr(a_scales), _ptr(masked_m), S, max_tokens, k_dim, n_dim, _ptr(w), _ptr(w_scales), num_w,
        _ptr(w_extra), _ptr(w_extra_scales), (MOE_E4M3 if fp8 else MOE_BF16) | (MOE_W_TILED if tiled else 0),
        epilogue, _ptr(out), _ptr(out_scales), _ptr(dev_status), _ptr(row_scale), _stream(stream)))
    return out, out_scales


def moe_grouped_gemm_combine(a, seg, w, src_row, inv_map, topk_w, max_tokens=0, shared_map=None, fq_scale=None,
                             a_scales=None, w_scales=None, w_extra=None, w_extra_scales=None, row_scale=None, y=None,
                             out=None, counters=None, dev_status=None, stream=None, tiled=False):
    """Down projection with the combine fused: a [rows, k] (or [S, max_tokens, k] with seg =
    masked_m and max_tokens > 0; else seg = cu_seqlens), w [num_w, H, k]; returns (out [T, H],
    y [rows, H], counters)."""
    _dev(a)
    fp8 = a.dtype == torch.uint8
    k_dim = a.shape[-1]
    rows = a.numel() // k_dim
    num_w, H = w.shape[0], w.shape[1]
    T, K = inv_map.shape
    nseg = seg.numel() if max_tokens else seg.numel() - 1
    if y is None:
        y = torch.empty(rows, H, dtype=torch.bfloat16, device=a.device)
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=a.device)
    if counters is None:
        counters = torch.zeros(T, H // 128, dtype=torch.int32, device=a.device)
    _check("moe_grouped_gemm_combine", lib().moe_grouped_gemm_combine(
        _ptr(a), _ptr(a_scales), _ptr(seg), nseg, max_tokens, rows, k_dim, H, _ptr(w), _ptr(w_scales), num_w,
        _ptr(w_extra), _ptr(w_extra_scales), (MOE_E4M3 if fp8 else MOE_BF16) | (MOE_W_TILED if tiled else 0),
        _ptr(y), _ptr(row_scale), _ptr(src_row), _ptr(inv_map), _ptr(topk_w), T, K, _ptr(shared_map),
        _ptr(fq_scale), _ptr(out), _ptr(counters), _ptr(dev_status), _stream(stream)))
    return out, y, counters


def moe_combine(y, inv_map, topk_w, shared_y=None, shared_map=None, fq_scale=None, out=None, stream=None):
    _dev(y)
    T, K = inv_map.shape
    H = y.shape[1]
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=y.device)
    _check("moe_combine", lib().moe_combine(_ptr(y), _ptr(inv_map), _ptr(topk_w), T, K, H, _ptr(shared_y),
                                            _ptr(shared_map), _ptr(fq_scale), _ptr(out), _stream(stream)))
    return out


def moe_combine_nvfp4(y, inv_map, topk_w, g_scale, shared_y=None, shared_map=None, out=None, stream=None):
    """Combine with the NVFP4 fake-quant of every routed row (g_scale: the per-tensor
    scale from moe_fq4_scale_from_amax)."""
    _dev(y)
    T, K = inv_map.shape
    H = y.shape[1]
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=y.device)
    _check("moe_combine_nvfp4", lib().moe_combine_nvfp4(_ptr(y), _ptr(inv_map), _ptr(topk_w), T, K, H,
                                                        _ptr(shared_y), _ptr(shared_map), _ptr(g_scale), _ptr(out),
                                                        _stream(stream)))
    return out


def moe_combine_verify(y, inv_map, topk_w, expected, dev_status, shared_y=None, shared_map=None, fq_scale=None,
                       stream=None):
    T, K = inv_map.shape
    H = y.shape[1]
    _check("moe_combine_verify", lib().moe_combine_verify(
        _ptr(y), _ptr(inv_map), _ptr(topk_w), T, K, H, _ptr(shared_y), _ptr(shared_map), _ptr(fq_scale),
        _ptr(expected), _ptr(dev_status), _stream(stream)))


def moe_combine_amax(y, inv_map, topk_w, amax, stream=None):
    T, K = inv_map.shape
    _check("moe_combine_amax", lib().moe_combine_amax(_ptr(y), _ptr(inv_map), _ptr(topk_w), T, K, y.shape[1],
                                                      _ptr(amax), _stream(stream)))
    return amax


def moe_amax_bf16(x, amax, stream=None):
    _dev(x)
    _check("moe_amax_bf16", lib().moe_amax_bf16(_ptr(x), x.numel(), _ptr(amax), _stream(stream)))
    return amax


def moe_fq_scale_from_amax(amax, scale=None, stream=None):
    if scale is None:
        scale = torch.empty(1, dtype=torch.float32, device=amax.device)
    _check("moe_fq_scale_from_amax", lib().moe_fq_scale_from_amax(_ptr(amax), _ptr(scale), _stream(stream)))
    return scale


def moe_fq4_scale_from_amax(amax, scale=None, stream=None):
    if scale is None:
        scale = torch.empty(1, dtype=torch.float32, device=amax.device)
    _check("moe_fq4_scale_from_amax", lib().moe_fq4_scale_from_amax(_ptr(amax), _ptr(scale), _stream(stream)))
    return scale


class MoeLayer:
    """Holds a layer's descriptor, weight pointers and workspace; forward() is one
    moe_layer_forward call.  Weights: w13 [E, 2I, H], w2 [E, H, I] (+ shared [2I, H],
    [H, I]) in BF16, or E4M3 codes with their 128x128 scales for dtype MOE_E4M3.
    weight_tiles=True: the layer keeps copies of the four weight tensors in the tile layout
    of moe_pack_weights (made once here) and computes from those."""

    def __init__(self, T, H, I, E, K, dtype=MOE_BF16, w13=None, w2=None, shared_w13=None, shared_w2=None,
                 w13_scales=None, w2_scales=None, shared_w13_scales=None, shared_w2_scales=None, device="cuda",
                 weight_in_down=False, max_tokens=0, fuse_combine=False, combine_fq="e4m3", dispatch_fq="e4m3",
                 gemm_pairs=False, weight_tiles=False):
        self.desc = LayerDesc(T, H, I, E, K, dtype, int(shared_w13 is not None), int(weight_in_down),
                              int(max_tokens), int(fuse_combine), _fmt(combine_fq), _fmt(dispatch_fq),
                              int(gemm_pairs), int(weight_tiles))
        if weight_tiles:
            w13, w2, shared_w13, shared_w2 = (None if t is None else moe_pack_weights(t)
                                              for t in (w13, w2, shared_w13, shared_w2))
        self.tensors = (w13, w2, shared_w13, shared_w2, w13_scales, w2_scales, shared_w13_scales, shared_w2_scales)
        self.weights = LayerWeights(_ptr(w13), _ptr(w13_scales), _ptr(w2), _ptr(w2_scales), _ptr(shared_w13),
                                    _ptr(shared_w13_scales), _ptr(shared_w2), _ptr(shared_w2_scales))
        nbytes = lib().moe_layer_workspace_bytes(ctypes.byref(self.desc))
        if nbytes == 0:
            raise MoeError("moe_layer_workspace_bytes", 1)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.views = LayerViews()
        _check("moe_layer_views", lib().moe_layer_views(ctypes.byref(self.desc), _ptr(self.ws),
                                                         ctypes.byref(self.views)))

    def view(self, name, shape, dtype):
        """A torch tensor over one workspace region (see LayerViews)."""
        ptr = getattr(self.views, name)
        n = 1
        for s in shape:
            n *= s
        base = _ptr(self.ws)
        off = ptr - base
        return self.ws[off:off + n * torch.empty(0, dtype=dtype).element_size()].view(dtype).view(*shape)

    def forward(self, x, out, topk_idx, topk_w, logits=None, num_tokens=None, fq_scale=None, dev_status=None,
                stream=None, dispatch_scale=None):
        _check("moe_layer_forward", lib().moe_layer_forward(
            ctypes.byref(self.desc), ctypes.byref(self.weights), _ptr(logits), _ptr(num_tokens), _ptr(topk_idx),
            _ptr(topk_w), _ptr(x), _ptr(fq_scale), _ptr(dispatch_scale), _ptr(out), _ptr(self.ws), self.ws.numel(),
            _ptr(dev_status), _stream(stream)))
        return out
