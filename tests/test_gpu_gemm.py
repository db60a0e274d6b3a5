"""GPU parity of the tcgen05 grouped GEMM (BF16 and E4M3 with 128-block scales; plain and
SwiGLU epilogues; BF16 also on pairs of SMs) against fp64 per-segment products computed by
the oracle side, on
ragged segments: empty segments, tails shorter than a tile, a partial 128-column tile,
the extra (shared-expert) segment, and more tiles than SMs so CTAs loop."""
import numpy as np
import pytest
import torch

import combine_moe_route_softmax_gb300 as moe
from gpu_helpers import bits, host, need_gpu
from oracle import moe_ref as ref
from oracle.formats import bf16_bits_to_f32, e4m3_decode

pytestmark = pytest.mark.gpu

SENTINEL = 0x7FC1   # a NaN pattern: rows outside every segment must keep it


def make_inputs(cu, rows_cap, k, n, num_w, extra, seed):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(rows_cap, k, generator=g).to(torch.bfloat16)
    w = (torch.randn(num_w, n, k, generator=g) / k ** 0.5).to(torch.bfloat16)
    wx = (torch.randn(n, k, generator=g) / k ** 0.5).to(torch.bfloat16) if extra else None
    return a, w, wx


def seg_weight(s, num_w, w, wx):
    return w[s] if s < num_w else wx


def reference(cu, a64, wlist, swiglu):
    out = []
    for s in range(len(cu) - 1):
        acc = a64[cu[s]:cu[s + 1]] @ wlist[s].T
        if swiglu:
            I = acc.shape[1] // 2
            g, u = acc[:, :I], acc[:, I:]
            with np.errstate(over="ignore"):
                acc = g / (1.0 + np.exp(-g)) * u
        out.append(acc)
    return np.concatenate(out) if out else None


CASES = [
    # cu_seqlens, rows_cap, k, n(weight rows), num_w, extra
    ([0, 5, 300, 300, 517, 700], 760, 256, 384, 4, True),
    ([0, 128, 256], 256, 128, 256, 2, False),
    ([0, 0, 1, 1], 8, 512, 512, 3, False),
    ([0, 2500, 5000], 5000, 512, 1024, 2, False),
    # ragged multi-tile segments (2, 4 and 4 M-tiles, the last holding 2 rows or 1 row) next
    # to a one-row segment
    ([0, 130, 130, 515, 1000, 1001], 1100, 256, 512, 4, True),
]


@pytest.mark.parametrize("pairs", [False, True], ids=["cta", "pairs"])
@pytest.mark.parametrize("swiglu", [False, True])
@pytest.mark.parametrize("case", CASES, ids=range(len(CASES)))
def test_bf16(case, swiglu, pairs):
    need_gpu()
    cu, rows_cap, k, n, num_w, extra = case
    if swiglu and n % 256:
        n += 128
    a, w, wx = make_inputs(cu, rows_cap, k, n, num_w, extra, seed=len(cu) + k)
    cols = n // 2 if swiglu else n
    out = torch.full((rows_cap, cols), SENTINEL, dtype=torch.int16).view(torch.bfloat16).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    moe.moe_grouped_gemm(a.cuda(), cu_t, w.cuda(), w_extra=None if wx is None else wx.cuda(),
                         epilogue=moe.MOE_EPI_SWIGLU if swiglu else moe.MOE_EPI_NONE, out=out, dev_status=st,
                         pairs=pairs)
    torch.cuda.synchronize()
    assert st.item() == 0
    f = lambda t: bf16_bits_to_f32(bits(t)).astype(np.float64)
    wl = [f(seg_weight(s, num_w, w, wx)) for s in range(len(cu) - 1)]
    want = reference(cu, f(a), wl, swiglu)
    got = f(out)
    N = cu[-1]
    if N:
        scale = np.abs(want).max()
        err = np.abs(got[:N] - want)
        assert np.all(err <= 2.0 ** -8 * np.abs(want) + 2e-3 * scale), err.max() / scale
    assert np.all(bits(out)[N:] == SENTINEL)


def quant_operands(a, w, wx):
    qa, sa = ref.act_quant_1x128(bf16_bits_to_f32(bits(a)))
    qw, sw = zip(*[ref.weight_quant_128x128(bf16_bits_to_f32(bits(w[i]))) for i in range(w.shape[0])])
    qx = sx = None
    if wx is not None:
        qx, sx = ref.weight_quant_128x128(bf16_bits_to_f32(bits(wx)))
    return qa, sa, np.stack(qw), np.stack(sw), qx, sx


@pytest.mark.parametrize("swiglu", [False, True])
@pytest.mark.parametrize("case", CASES, ids=range(len(CASES)))
def test_e4m3_block_scaled(case, swiglu):
    need_gpu()
    cu, rows_cap, k, n, num_w, extra = case
    if swiglu and n % 256:
        n += 128
    a, w, wx = make_inputs(cu, rows_cap, k, n, num_w, extra, seed=len(cu) + k + 1)
    qa, sa, qw, sw, qx, sx = quant_operands(a, w, wx)
    T = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()
    cols = n // 2 if swiglu else n
    if swiglu:
        out = torch.zeros(rows_cap, cols, dtype=torch.uint8, device="cuda")
        out_s = torch.full((rows_cap, cols // 128), -1.0, dtype=torch.float32, device="cuda")
    else:
        out = torch.full((rows_cap, cols), SENTINEL, dtype=torch.int16).view(torch.bfloat16).cuda()
        out_s = None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    moe.moe_grouped_gemm(T(qa), cu_t, T(qw), a_scales=T(sa), w_scales=T(sw), w_extra=T(qx), w_extra_scales=T(sx),
                         epilogue=moe.MOE_EPI_SWIGLU if swiglu else moe.MOE_EPI_NONE, out=out, out_scales=out_s,
                         dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    a64 = ref.dequant(qa, sa, 1)
    wl = [ref.dequant(qw[s], sw[s], 128) if s < num_w else ref.dequant(qx, sx, 128) for s in range(len(cu) - 1)]
    want = reference(cu, a64, wl, swiglu)
    N = cu[-1]
    if not N:
        return
    scale = np.abs(want).max()
    if not swiglu:
        got = bf16_bits_to_f32(bits(out)).astype(np.float64)
        err = np.abs(got[:N] - want)
        assert np.all(err <= 2.0 ** -8 * np.abs(want) + 2e-3 * scale), err.max() / scale
        assert np.all(bits(out)[N:] == SENTINEL)
    else:
        gq, gs = host(out)[:N], host(out_s)[:N]
        # scales: amax/448 of each 1x128 block of h (up to the accumulation error)
        amax = np.abs(want.reshape(N, -1, 128)).max(axis=-1)
        ws = np.where(amax > 0, amax / 448.0, 1.0)
        assert np.allclose(gs, ws, rtol=1e-3, atol=1e-30)
        got = e4m3_decode(gq).astype(np.float64) * np.repeat(gs.astype(np.float64), 128, axis=1)
        srep = np.repeat(gs.astype(np.float64), 128, axis=1)
        err = np.abs(got - want)
        assert np.all(err <= 2.0 ** -4 * np.abs(want) * 1.01 + srep * 2.0 ** -9 + 1e-3 * scale)
        assert np.all(host(out_s)[N:] == -1.0)


def streamed_counts(seed, n_big, big_rows, n_small):
    """Segment lengths: n_small segments of 1..32 rows (some empty) among n_big large ones."""
    rng = np.random.default_rng(seed)
    counts = list(rng.integers(0, 33, n_small)) + [big_rows + int(rng.integers(0, 100)) for _ in range(n_big)]
    rng.shuffle(counts)
    return [int(c) for c in counts]


STREAM_CASES = [
    # swiglu, layout, n (weight rows), big segments, their rows, k
    (True, "contiguous", 4096, 9, 2000, 256),      # 16 N-tiles
    (False, "contiguous", 2048, 10, 3900, 256),    # 8 N-tiles
    (True, "batched", 4096, 12, 900, 256),
    (False, "batched", 2048, 34, 900, 256),
    (True, "contiguous", 2816, 10, 2100, 256),     # 11 N-tiles: an odd N-tile count
    (False, "contiguous", 2176, 10, 3000, 256),    # 9 N-tiles, the last one half outside the weights
]


@pytest.mark.parametrize("pairs", [False, True], ids=["cta", "pairs"])
@pytest.mark.parametrize("swiglu,layout,n,n_big,big_rows,k", STREAM_CASES,
                         ids=[f"{'swiglu' if c[0] else 'plain'}-{c[1]}-n{c[2]}-k{c[5]}" for c in STREAM_CASES])
def test_bf16_short_segments_on_streaming_ctas(swiglu, layout, n, n_big, big_rows, k, pairs):
    """Enough units per CTA that the launch splits its CTAs: segments of at most 32 rows go
    to streaming CTAs (weights as the MMA's M operand, the segment's rows as N = 32), the
    rest to the MMA pipeline.  Covers a short extra (shared-expert) segment, empty segments,
    row_scale on the plain epilogue, the batched layout's masked_m bounds, odd N-tile counts
    and a last N-tile that reaches past the weight rows."""
    need_gpu()
    counts = streamed_counts(7 + swiglu + 2 * (layout == "batched") + n, n_big, big_rows, 60)
    counts.append(20)                   # the extra segment, short: streamed from w_extra
    num_w = len(counts) - 1
    S = len(counts)
    g = torch.Generator().manual_seed(11)
    w = (torch.randn(num_w, n, k, generator=g) / k ** 0.5).to(torch.bfloat16)
    wx = (torch.randn(n, k, generator=g) / k ** 0.5).to(torch.bfloat16)
    cols = n // 2 if swiglu else n
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    f = lambda b: bf16_bits_to_f32(b).astype(np.float64)
    epi = moe.MOE_EPI_SWIGLU if swiglu else moe.MOE_EPI_NONE
    if layout == "contiguous":
        cu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        rows = int(cu[-1])
        a = torch.randn(rows, k, generator=g).to(torch.bfloat16)
        rs = None if swiglu else torch.rand(rows, generator=g) + 0.5
        out = torch.full((rows, cols), SENTINEL, dtype=torch.int16).view(torch.bfloat16).cuda()
        moe.moe_grouped_gemm(a.cuda(), torch.from_numpy(cu).cuda(), w.cuda(), w_extra=wx.cuda(), epilogue=epi,
                             out=out, dev_status=st, row_scale=None if rs is None else rs.cuda(), pairs=pairs)
        spans = [(int(cu[s]), int(cu[s + 1]), int(cu[s + 1])) for s in range(S)]
    else:
        if pairs:
            pytest.skip("the pair computation takes contiguous segments")
        mt = 1024
        a = torch.randn(S, mt, k, generator=g).to(torch.bfloat16)
        rs = None if swiglu else torch.rand(S * mt, generator=g) + 0.5
        out = torch.full((S, mt, cols), SENTINEL, dtype=torch.int16).view(torch.bfloat16).cuda()
        moe.moe_grouped_gemm_batched(a.cuda(), torch.tensor(counts, dtype=torch.int32).cuda(), w.cuda(),
                                     w_extra=wx.cuda(), epilogue=epi, out=out, dev_status=st,
                                     row_scale=None if rs is None else rs.cuda())
        spans = [(s * mt, s * mt + counts[s], (s + 1) * mt) for s in range(S)]
    torch.cuda.synchronize()
    assert st.item() == 0
    ob = bits(out).reshape(-1, cols)
    ab = bits(a).reshape(-1, k)
    w64, wx64 = f(bits(w)), f(bits(wx))
    for s, (b, e, cap) in enumerate(spans):
        assert np.all(ob[e:cap] == SENTINEL)          # rows past a batched segment's count
        if e == b:
            continue
        acc = f(ab[b:e]) @ (w64[s] if s < num_w else wx64).T
        if swiglu:
            I = acc.shape[1] // 2
            with np.errstate(over="ignore"):
                acc = acc[:, :I] / (1.0 + np.exp(-acc[:, :I])) * acc[:, I:]
        elif rs is not None:
            acc = acc * rs.numpy().astype(np.float64)[b:e, None]
        scale = np.abs(acc).max()
        err = np.abs(f(ob[b:e]) - acc)
        assert np.all(err <= 2.0 ** -8 * np.abs(acc) + 2e-3 * scale), (s, e - b, err.max() / scale)


@pytest.mark.parametrize("swiglu", [False, True])
def test_pairs_and_single_cta_agree_bit_for_bit(swiglu):
    """The two BF16 computations accumulate the same products in the same order: identical
    output on a mix of long, ragged and streamed segments."""
    need_gpu()
    k, n = 512, 1024
    counts = streamed_counts(3, 12, 1500, 80)
    cu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    g = torch.Generator().manual_seed(21)
    a = torch.randn(int(cu[-1]), k, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(len(counts), n, k, generator=g) / k ** 0.5).to(torch.bfloat16).cuda()
    epi = moe.MOE_EPI_SWIGLU if swiglu else moe.MOE_EPI_NONE
    cu_t = torch.from_numpy(cu).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o1, _ = moe.moe_grouped_gemm(a, cu_t, w, epilogue=epi, dev_status=st)
    o2, _ = moe.moe_grouped_gemm(a, cu_t, w, epilogue=epi, dev_status=st, pairs=True)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


@pytest.mark.parametrize("swiglu,n,n_big,big_rows,k", [(True, 4096, 9, 2000, 256), (False, 2048, 10, 3900, 384)])
def test_pairs_and_single_cta_agree_bit_for_bit_when_streaming(swiglu, n, n_big, big_rows, k):
    """With segments of at most 32 rows on the streaming CTAs of both computations: the
    streamed products are summed in the same order too (even and odd K blocks apart, then
    added)."""
    need_gpu()
    counts = streamed_counts(31 + k, n_big, big_rows, 60)
    cu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    g = torch.Generator().manual_seed(23)
    a = torch.randn(int(cu[-1]), k, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(len(counts), n, k, generator=g) / k ** 0.5).to(torch.bfloat16).cuda()
    epi = moe.MOE_EPI_SWIGLU if swiglu else moe.MOE_EPI_NONE
    cu_t = torch.from_numpy(cu).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o1, _ = moe.moe_grouped_gemm(a, cu_t, w, epilogue=epi, dev_status=st)
    o2, _ = moe.moe_grouped_gemm(a, cu_t, w, epilogue=epi, dev_status=st, pairs=True)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
