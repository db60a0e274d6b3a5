"""GPU parity of the tcgen05 grouped GEMM (BF16 and E4M3 with 128-block scales; plain and
SwiGLU epilogues) against fp64 per-segment products computed by the oracle side, on
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
    # CTA pairs on two M-tiles of one weight tile (2, 4 and 4 M-tiles, the second of a pair
    # holding 2 rows or 1 row) next to a one-row segment (a pair of N-tiles)
    ([0, 130, 130, 515, 1000, 1001], 1100, 256, 512, 4, True),
]


@pytest.mark.parametrize("swiglu", [False, True])
@pytest.mark.parametrize("case", CASES, ids=range(len(CASES)))
def test_bf16(case, swiglu):
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
                         epilogue=moe.MOE_EPI_SWIGLU if swiglu else moe.MOE_EPI_NONE, out=out, dev_status=st)
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
