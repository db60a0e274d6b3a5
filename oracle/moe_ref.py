"""Plain CPU oracle of the single-GPU MoE layer: route, permute, experts, combine.

Test infrastructure only (see the package docstring).  Every step is the plain
definition, written out with numpy; library primitives (argsort, matmul, exp) serve as
steps, with no blocking or fusion beyond what the definition states.

Notation follows the pages: T tokens, H hidden size, I expert intermediate size,
E routed experts, K = experts per token (top-k), topk_idx / topk_weights [T, K],
cu_seqlens over expert segments, and the expert-major row layout [NvS, H] of the
MoonEP page (after dispatch the rows arrive grouped by expert).
"""
import numpy as np

from .formats import (bf16_bits_to_f32, e2m1_decode, e2m1_encode, e4m3_decode, e4m3_decode64, e4m3_encode,
                      f32_to_bf16_bits)

F32 = np.float32
STATUS_BAD_EXPERT = 1
STATUS_VERIFY_MISMATCH = 2
STATUS_OVERFLOW = 8


# ----------------------------------------------------------------------------- route
def route_topk(logits, K, num_tokens=None):
    """Router: softmax over the E experts, top-K, renormalise over the chosen K.

    The DeepEP page passes per-token ``topk_weights`` / ``topk_ids`` into dispatch and
    the MoonEP page works with [T, K] expert ids, but neither defines the router
    function; this takes the plain softmax -> top-k -> renormalise reading.  Softmax is
    computed in fp64; the top K are chosen on the float32 logits (softmax is monotone, so this is the
    same set) in descending order, ties going to the lower expert id; the chosen
    probabilities are divided by their sum and rounded once to float32.

    Rows t >= num_tokens are padding: ids -1, weights 0 (the power-of-two receive
    bucket of the permute-scratch page pads the token count and marks the extra rows
    with topk_idx = -1).
    """
    logits = np.asarray(logits, dtype=F32)
    T, E = logits.shape
    n = T if num_tokens is None else int(num_tokens)
    idx = np.full((T, K), -1, dtype=np.int32)
    w = np.zeros((T, K), dtype=F32)
    ids = np.arange(E)
    for t in range(min(n, T)):
        l64 = logits[t].astype(np.float64)
        p = np.exp(l64 - l64.max())
        p = p / p.sum()
        order = np.lexsort((ids, -logits[t]))      # primary: logit desc; then id asc
        sel = order[:K]
        idx[t] = sel
        w[t] = (p[sel] / p[sel].sum()).astype(F32)
    return idx, w


# --------------------------------------------------------------------------- permute
def permute(topk_idx, E, with_shared=False):
    """Counting sort of the valid (token, slot) pairs into the expert-major layout.

    MoonEP page: after dispatch the rows are laid out expert by expert as [NvS, H]
    with cu_seqlens marking the segments, and the experts run as a grouped GEMM over
    those segments.  Flat slot s = t*K + k.  Segment e holds, in ascending s, every
    slot with topk_idx == e (a stable sort by expert id).  Slots with topk_idx == -1 are padding
    and get no row (the Mega-MoE page's ``valid = topk_idx >= 0`` mask).  An id outside
    [-1, E) is a data error: status bit 0 is set and the slot is treated as padding.

    with_shared appends one more segment (index E) for the shared expert: every token
    with at least one valid slot, in ascending t, its source index being T*K + t.
    (On the Mega-MoE page a fused shared expert occupies the combine's final slot; here
    it runs as one extra dense segment of the same grouped GEMM, like the extra
    [E, E+B) segments of the MoonEP layout.)

    Returns cu_seqlens [E+1 or E+2] (leading 0), src_row [cap] (row -> source index,
    -1 beyond the last row), inv_map [T, K] (slot -> row or -1), shared_map [T] (token ->
    shared row or -1; None without with_shared) and the status word.  cap = T*K (+T), the
    bound taken from the inputs, as the permute-scratch page requires.
    """
    topk_idx = np.asarray(topk_idx, dtype=np.int32)
    T, K = topk_idx.shape
    flat = topk_idx.reshape(-1)
    bad = (flat >= E) | (flat < -1)
    status = STATUS_BAD_EXPERT if bad.any() else 0
    valid = (flat >= 0) & (flat < E)
    segments = [np.nonzero(valid & (flat == e))[0] for e in range(E)]
    if with_shared:
        tok_valid = valid.reshape(T, K).any(axis=1)
        segments.append(T * K + np.nonzero(tok_valid)[0])
    counts = np.array([len(s) for s in segments], dtype=np.int64)
    cu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    cap = T * K + (T if with_shared else 0)
    n_total = int(cu[-1])
    src_row = np.full(cap, -1, dtype=np.int32)
    if n_total:
        src_row[:n_total] = np.concatenate(segments)
    n_routed = int(cu[E])
    inv_map = np.full(T * K, -1, dtype=np.int32)
    inv_map[src_row[:n_routed]] = np.arange(n_routed, dtype=np.int32)
    shared_map = None
    if with_shared:
        shared_map = np.full(T, -1, dtype=np.int32)
        shared_map[src_row[n_routed:n_total] - T * K] = np.arange(n_routed, n_total, dtype=np.int32)
    return cu, src_row, inv_map.reshape(T, K), shared_map, status


def permute_batched(topk_idx, E, max_tokens, with_shared=False):
    """The expert-batched layout of the DeepEP page: each expert gets a fixed block of
    max_tokens rows ([E, max_tokens, H], 3-D) plus the number of rows it really received,
    where the high-throughput path uses the contiguous 2-D layout.

    The page does not fix the order of the rows inside a block; this takes the order of
    the contiguous layout: block e lists, in ascending flat slot s = t*K + k, the slots with
    topk_idx == e, so its row r is the r-th such slot.  With with_shared, block E lists
    the tokens that have a valid slot, ascending t, source index T*K + t.  A block keeps
    its first max_tokens entries; the others are dropped (no row, inv_map / shared_map -1)
    and set the overflow bit of the status word.  An id outside [-1, E) is padding with
    the bad-expert bit, as in the contiguous permute.

    Returns masked_m [nseg] (rows kept per block), src_row [nseg * max_tokens] (source of
    each row, -1 for unused rows), inv_map [T, K], shared_map [T] (None without
    with_shared) and the status word.
    """
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, K = idx.shape
    nseg = E + (1 if with_shared else 0)
    status = 0
    blocks = [[] for _ in range(nseg)]
    for t in range(T):
        for k in range(K):
            e = int(idx[t, k])
            if e == -1:
                continue
            if e < -1 or e >= E:
                status |= STATUS_BAD_EXPERT
                continue
            blocks[e].append(t * K + k)
    if with_shared:
        blocks[E] = [T * K + t for t in range(T) if any(0 <= int(e) < E for e in idx[t])]
    masked_m = np.zeros(nseg, dtype=np.int32)
    src_row = np.full(nseg * max_tokens, -1, dtype=np.int32)
    inv_map = np.full((T, K), -1, dtype=np.int32)
    shared_map = np.full(T, -1, dtype=np.int32) if with_shared else None
    for b, entries in enumerate(blocks):
        if len(entries) > max_tokens:
            status |= STATUS_OVERFLOW
        kept = entries[:max_tokens]
        masked_m[b] = len(kept)
        for r, src in enumerate(kept):
            row = b * max_tokens + r
            src_row[row] = src
            if src < T * K:
                inv_map[src // K, src % K] = row
            else:
                shared_map[src - T * K] = row
    return masked_m, src_row, inv_map, shared_map, status


def row_tokens(src_row, T, K):
    """Token of each permuted row (-1 for rows past the last one)."""
    src_row = np.asarray(src_row, dtype=np.int64)
    tok = np.where(src_row < T * K, src_row // K, src_row - T * K)
    return np.where(src_row < 0, -1, tok)


def gather_rows(x_bits, src_row, T, K):
    """Xp[p] = x[token(p)]: an exact copy of each routed token's BF16 row (rows past the
    last one are left zero; the GPU path leaves them untouched)."""
    tok = row_tokens(src_row, T, K)
    out = np.zeros((len(src_row), x_bits.shape[1]), dtype=np.uint16)
    ok = tok >= 0
    out[ok] = x_bits[tok[ok]]
    return out


# ------------------------------------------------------------------------ FP8 blocks
def _block_scale(amax):
    """s = amax / 448 in float32; 1 where that is not positive (an all-zero block)."""
    s = (np.asarray(amax, dtype=F32) / F32(448.0)).astype(F32)
    return np.where(s > 0, s, F32(1.0)).astype(F32)


def act_quant_1x128(x):
    """Per-row, per-128-column FP8 quantisation of activations.

    The DeepEP page's low-latency dispatch can quantise BF16 tokens to FP8 itself,
    sending codes plus scales that the receiver dequantises; its DeepGEMM test sizes
    tiles by block_n x block_k.
    The scale format is not stated; this takes an FP32 scale per 1x128 block,
    s = amax / 448, and codes q = e4m3(x / s) (round to nearest even, saturating), with
    the divisions in float32.  Dequantisation is q * s.
    Returns (codes uint8 [R, C], scales float32 [R, C/128]).
    """
    x = np.asarray(x, dtype=F32)
    R, C = x.shape
    assert C % 128 == 0
    xb = x.reshape(R, C // 128, 128)
    s = _block_scale(np.abs(xb).max(axis=-1))
    q = e4m3_encode((xb / s[..., None]).astype(F32))
    return q.reshape(R, C), s


def weight_quant_128x128(w):
    """FP8 quantisation of a weight matrix [N, K] with one FP32 scale per 128x128 block
    (the block_n x block_k weight tiles of the DeepEP page's DeepGEMM test), same rule as above.
    Returns (codes uint8 [N, K], scales float32 [N/128, K/128])."""
    w = np.asarray(w, dtype=F32)
    N, K = w.shape
    assert N % 128 == 0 and K % 128 == 0
    wb = w.reshape(N // 128, 128, K // 128, 128)
    s = _block_scale(np.abs(wb).max(axis=(1, 3)))
    q = e4m3_encode((wb / s[:, None, :, None]).astype(F32))
    return q.reshape(N, K), s


def dequant(codes, scales, block_rows):
    """codes * scale in float64, the scale block being block_rows x 128."""
    R, C = codes.shape
    v = e4m3_decode64(codes).reshape(R // block_rows, block_rows, C // 128, 128)
    v *= scales.astype(np.float64)[:, None, :, None]
    return v.reshape(R, C)


# --------------------------------------------------------------------------- experts
def swiglu_expert(x, w13, w2):
    """One SwiGLU expert in fp64: y = W_down (silu(W_gate x) * (W_up x)).

    Gate and up are the two halves of the fused ``w1`` of the DeepEP page ([2n, k]
    with gate rows first); the MoonEP page runs the same three projections (gate, up,
    down) as grouped GEMMs.  silu(z) = z / (1 + e^-z).
    x [m, H], w13 [2I, H], w2 [H, I] -> [m, H].
    """
    x = np.asarray(x, dtype=np.float64)
    I = w13.shape[0] // 2
    g = x @ np.asarray(w13[:I], dtype=np.float64).T
    u = x @ np.asarray(w13[I:], dtype=np.float64).T
    with np.errstate(over="ignore"):
        h = g / (1.0 + np.exp(-g)) * u
    return h @ np.asarray(w2, dtype=np.float64).T


def qdq_f32(r, s):
    """Combine fake-quant of one router-weighted row (Mega-MoE page: combine_quantizer
    fake-quantises the router-weighted per-(token, slot) rows with a constant global
    scale).  In float32: t = r * s, snapped to E4M3 (nearest even, saturating), then
    divided by s."""
    s = F32(s)
    t = (np.asarray(r, dtype=F32) * s).astype(F32)
    q = e4m3_decode(e4m3_encode(t))
    return (q / s).astype(F32)


NVFP4_BLOCK = 16


def nvfp4_qdq_f32(r, g):
    """NVFP4 fake-quant of router-weighted rows (the Mega-MoE page runs its combine and
    dispatch quantisers with NVFP4 units as well as FP8 ones, and leaves the format's
    arithmetic to that recipe; this is the two-level NVFP4 reading).  r [..., H] float32,
    H a multiple of 16; g the float32 per-tensor scale (448 * 6 / calibration amax).
    For each block of 16 consecutive elements along the last axis, in float32:
      a = max |r| over the block;
      block scale code s_b = e4m3(fl32(fl32(a / 6) * g)) (nearest even, saturating);
      inv = fl32(g / e4m3_decode(s_b)) (0 when s_b decodes to 0),
      d   = fl32(e4m3_decode(s_b) / g);
      each element: q = e2m1(fl32(r * inv)) (nearest even, saturating at 6),
                    r' = fl32(e2m1_decode(q) * d).
    Returns r' (float32, the shape of r)."""
    r = np.asarray(r, dtype=F32)
    g = F32(g)
    blocks = r.reshape(r.shape[:-1] + (r.shape[-1] // NVFP4_BLOCK, NVFP4_BLOCK))
    a = np.abs(blocks).max(axis=-1, keepdims=True).astype(F32)
    sf = ((a / F32(6.0)).astype(F32) * g).astype(F32)
    sdec = e4m3_decode(e4m3_encode(sf))
    with np.errstate(divide="ignore"):
        inv = np.where(sdec > 0, (g / np.where(sdec > 0, sdec, F32(1.0))).astype(F32), F32(0.0)).astype(F32)
    d = (sdec / g).astype(F32)
    q = e2m1_decode(e2m1_encode((blocks * inv).astype(F32)))
    return (q * d).astype(F32).reshape(r.shape)


def nvfp4_scale_from_amax(amax):
    """Per-tensor NVFP4 scale 448 * 6 / amax in float32 (1 when amax is 0): the largest
    block (amax / 6) maps onto the largest E4M3 block scale, 448."""
    amax = F32(amax)
    return F32(F32(2688.0) / amax) if amax > 0 else F32(1.0)


# ------------------------------------------------------------------- dispatch fake-quant
def dispatch_qdq_bits(x_bits, s, fmt="e4m3"):
    """Dispatch fake-quant of BF16 token rows (Mega-MoE page: the dispatch quantiser
    fake-quantises the tokens the experts receive, with a calibrated or constant global
    scale).  E4M3: in float32, t = x * s, snapped to E4M3 (nearest even, saturating),
    divided by s.  NVFP4 (fmt "nvfp4", the page's other unit): nvfp4_qdq_f32(x, s) with s
    the per-tensor scale.  Either way rounded back to BF16 -- the experts' input type
    here.  Returns BF16 bits."""
    x = bf16_bits_to_f32(np.asarray(x_bits, dtype=np.uint16))
    return f32_to_bf16_bits(nvfp4_qdq_f32(x, s) if fmt == "nvfp4" else qdq_f32(x, s))


def tensor_amax(x_bits):
    """Calibration of the dispatch scale: the largest |x| of a BF16 tensor (float32)."""
    x = bf16_bits_to_f32(np.asarray(x_bits, dtype=np.uint16))
    return F32(np.abs(x).max()) if x.size else F32(0.0)


# --------------------------------------------------------------------------- combine
def combine(y_bits, inv_map, topk_w, shared_bits=None, shared_map=None, fq_scale=None, fq_format="e4m3"):
    """Fixed-order combine (Mega-MoE page): per token, the valid slots in ascending
    order, each row router-weighted (float32 product of the BF16 row and the float32
    weight) and optionally fake-quantised, summed in float32 starting from +0, then the
    shared expert's row (unquantised) last, then one rounding to BF16.

    y_bits [R, H] uint16: expert output rows in the permuted layout; row of slot (t, k)
    is inv_map[t, k] (-1: padding, skipped).  Shared row of token t: shared_bits[t]
    (dense) or shared_bits[shared_map[t]].  A token with no valid slot is a padding
    token: out = +0 and no shared row is added.
    topk_w None: the rows are already router-weighted (the MoonEP page applies the route
    weights inside the expert computation, before the down projection's output is
    combined, so the combine only sums), and r = float(y).
    fq_format: "e4m3" (qdq_f32 with the scale fq_scale) or "nvfp4" (nvfp4_qdq_f32 with the
    per-tensor scale fq_scale).
    Returns out bits [T, H] uint16.
    """
    inv_map = np.asarray(inv_map)
    T, K = inv_map.shape
    H = y_bits.shape[1]
    acc = np.zeros((T, H), dtype=F32)
    any_valid = (inv_map >= 0).any(axis=1)
    for k in range(K):
        rows = inv_map[:, k]
        ok = rows >= 0
        y = bf16_bits_to_f32(y_bits[np.where(ok, rows, 0)])
        if topk_w is None:
            r = y
        else:
            r = (y * np.asarray(topk_w, dtype=F32)[:, k:k + 1]).astype(F32)
        if fq_scale is not None:
            r = nvfp4_qdq_f32(r, fq_scale) if fq_format == "nvfp4" else qdq_f32(r, fq_scale)
        acc = np.where(ok[:, None], (acc + r).astype(F32), acc)
    if shared_bits is not None:
        srow = np.arange(T) if shared_map is None else np.asarray(shared_map)
        use = any_valid & (srow >= 0)
        ys = bf16_bits_to_f32(shared_bits[np.where(use, srow, 0)])
        acc = np.where(use[:, None], (acc + ys).astype(F32), acc)
    return f32_to_bf16_bits(acc)


def combine_amax(y_bits, inv_map, topk_w):
    """Calibration (max calibration on the Mega-MoE page): the largest |r| over every
    valid router-weighted row element r = float32(y * w).  0 if there is no valid slot."""
    inv_map = np.asarray(inv_map)
    best = F32(0.0)
    for k in range(inv_map.shape[1]):
        rows = inv_map[:, k]
        ok = rows >= 0
        if not ok.any():
            continue
        y = bf16_bits_to_f32(y_bits[rows[ok]])
        r = y if topk_w is None else (y * np.asarray(topk_w, dtype=F32)[ok, k:k + 1]).astype(F32)
        best = max(best, F32(np.abs(r).max()))
    return F32(best)


def fq_scale_from_amax(amax):
    """Constant combine scale 448 / amax in float32 (1 when amax is 0)."""
    amax = F32(amax)
    return F32(F32(448.0) / amax) if amax > 0 else F32(1.0)


# ----------------------------------------------------------------- layer reference
def _f64_weights(w_bits_or_f):
    w = np.asarray(w_bits_or_f)
    if w.dtype == np.uint16:
        return bf16_bits_to_f32(w).astype(np.float64)
    return w.astype(np.float64)


def layer_reference(x_bits, topk_idx, topk_w, w13, w2, shared=None, tokens=None,
                    fq_scale=None, fp8=False, dispatch_scale=None, fq_format="e4m3", dispatch_format="e4m3",
                    workers=None):
    """Dense per-token reference MoE in fp64 (the MoonEP page validates its path by
    comparing with a straightforward per-token MoE): for each token, for the valid slots in ascending
    order, r = w_k * expert_{idx_k}(x_t) (optionally fake-quantised as in the combine);
    the sum of the r, plus the shared expert's output when the token has a valid slot.
    No final rounding: the result is the float64 value the BF16 output approximates.

    x_bits [T, H] uint16 BF16; w13 [E, 2I, H], w2 [E, H, I] (uint16 BF16 bits, or float
    arrays); shared = (w13_s [2I, H], w2_s [H, I]) or None; tokens: subset of token
    indices (default all).  fp8=True runs the experts on FP8-quantised operands as the
    FP8 path defines them: x and h quantised per 1x128 block, weights per 128x128 block,
    all dequantised to fp64 (the tighter reference for the FP8 configuration).
    dispatch_scale: the routed experts see dispatch_qdq_bits(x, s) instead of x; the
    shared expert keeps the original x (the Mega-MoE page requires the shared expert to be
    unfused when the dispatch is quantised, since a fused one would read the same tokens).
    fq_format: the combine fake-quant's format when fq_scale is given, "e4m3" or "nvfp4";
    dispatch_format: the dispatch fake-quant's, likewise.
    workers: how many experts to compute at once in threads (default 1); the result does
    not depend on it.
    Returns float64 [len(tokens), H].
    """
    x = bf16_bits_to_f32(np.asarray(x_bits)).astype(np.float64)
    T, H = x.shape
    topk_idx = np.asarray(topk_idx)
    K = topk_idx.shape[1]
    toks = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)

    def prep_x(rows):
        if not fp8:
            return rows
        q, s = act_quant_1x128(rows.astype(F32))
        return dequant(q, s, 1)

    def prep_w(wm):
        if not fp8:
            return _f64_weights(wm)
        wm = np.asarray(wm)
        q, s = weight_quant_128x128(bf16_bits_to_f32(wm) if wm.dtype == np.uint16 else wm.astype(F32))
        return dequant(q, s, 128)

    def run_expert(xr, w13e, w2e):
        if not fp8:
            return swiglu_expert(xr, w13e, w2e)
        I = w13e.shape[0] // 2
        g = xr @ w13e[:I].T
        u = xr @ w13e[I:].T
        with np.errstate(over="ignore"):
            h = (g / (1.0 + np.exp(-g)) * u).astype(F32)
        qh, sh = act_quant_1x128(h)
        return dequant(qh, sh, 1) @ w2e.T

    xs = prep_x(x[toks])
    xs_shared = xs
    if dispatch_scale is not None:
        xq = dispatch_qdq_bits(np.asarray(x_bits)[toks], dispatch_scale, dispatch_format)
        xs = prep_x(bf16_bits_to_f32(xq).astype(np.float64))
    # expert outputs for every (token, slot) pair of the subset, expert by expert; the experts
    # are independent, so up to `workers` of them run at once in threads (numpy's array
    # operations release the interpreter lock), each computed exactly as when run alone
    contrib = np.zeros((len(toks), K, H), dtype=np.float64)
    sub_idx = topk_idx[toks]

    def expert_rows(e):
        where = np.nonzero(sub_idx == e)
        return where, run_expert(xs[where[0]], prep_w(w13[e]), prep_w(w2[e]))

    experts = np.unique(sub_idx[sub_idx >= 0])
    n_workers = min(len(experts), workers if workers else 1)
    if n_workers > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(n_workers) as pool:
            results = list(pool.map(expert_rows, experts))
    else:
        results = [expert_rows(e) for e in experts]
    for where, ye in results:
        contrib[where[0], where[1]] = ye
    out = np.zeros((len(toks), H), dtype=np.float64)
    wsub = np.asarray(topk_w, dtype=F32)[toks]
    for k in range(K):
        ok = sub_idx[:, k] >= 0
        r = wsub[:, k:k + 1].astype(np.float64) * contrib[:, k]
        if fq_scale is not None:
            rq = nvfp4_qdq_f32 if fq_format == "nvfp4" else qdq_f32
            r = rq(r.astype(F32), fq_scale).astype(np.float64)
        out = np.where(ok[:, None], out + r, out)
    if shared is not None:
        any_valid = (sub_idx >= 0).any(axis=1)
        if any_valid.any():
            ys = run_expert(xs_shared[any_valid], prep_w(shared[0]), prep_w(shared[1]))
            out[any_valid] += ys
    return out


def max_rel_err(y, ref):
    """max |y - ref| / max |ref| (the layer's tolerance metric)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    return float(np.abs(y - ref).max() / (den if den > 0 else 1.0))
