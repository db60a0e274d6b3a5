"""The tiled weight layout (moe_pack_weights, MOE_W_TILED, moe_layer_desc_t.weight_tiles):
the packed bytes follow the layout the header defines, restated here with numpy, and every
grouped GEMM call and layer configuration that reads tiled weights returns exactly what the
row-major call returns (the same products accumulated in the same order, from the same
weight bytes fetched in another order), on ragged, streamed, batched, fused and E4M3 cases.
Parity of the row-major computation with the oracle is checked in test_gpu_gemm.py and
test_gpu_layer.py, and the full-size layer parity there runs on tiled weights, as the
benchmark does."""
import numpy as np
import pytest
import torch

import combine_moe_route_softmax_gb300 as moe
from combine_moe_route_softmax_gb300 import synth
from combine_moe_route_softmax_gb300.synth import WORKLOADS, scaled
from gpu_helpers import bits, host, need_gpu
from test_gpu_gemm import CASES, STREAM_CASES, make_inputs, streamed_counts

pytestmark = pytest.mark.gpu


def tiles_by_definition(raw, E, N, K_bytes):
    """Bytes of [E, N, K_bytes] in the documented order: box (e, nb, kb) = rows
    [128 nb, 128 nb + 128) of matrix e, bytes [128 kb, 128 kb + 128) of each row, boxes in
    (e, nb, kb) order, each box's rows in order."""
    out = np.empty(E * N * K_bytes, dtype=np.uint8)
    pos = 0
    for e in range(E):
        for nb in range(N // 128):
            for kb in range(K_bytes // 128):
                box = raw[e, 128 * nb:128 * nb + 128, 128 * kb:128 * kb + 128]
                out[pos:pos + box.size] = box.reshape(-1)
                pos += box.size
    return out


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_pack_follows_the_documented_layout(dtype):
    need_gpu()
    E, N, K = 3, 384, 512
    g = torch.Generator().manual_seed(5)
    if dtype == "bf16":
        w = torch.randn(E, N, K, generator=g).to(torch.bfloat16).cuda()
    else:
        w = torch.randint(0, 256, (E, N, K), generator=g, dtype=torch.uint8).cuda()
    t = moe.moe_pack_weights(w)
    torch.cuda.synchronize()
    raw = host(w.view(torch.uint8)).reshape(E, N, -1)
    want = tiles_by_definition(raw, E, N, raw.shape[2])
    assert np.array_equal(host(t.view(torch.uint8)).reshape(-1), want)
    # one matrix (the shared expert's form)
    t1 = moe.moe_pack_weights(w[1])
    torch.cuda.synchronize()
    assert np.array_equal(host(t1.view(torch.uint8)).reshape(-1), tiles_by_definition(raw[1:2], 1, N, raw.shape[2]))


def same_bits(x, y):
    return np.array_equal(bits(x), bits(y)) if x.dtype != torch.uint8 else torch.equal(x, y)


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("swiglu", [False, True])
@pytest.mark.parametrize("case", CASES, ids=range(len(CASES)))
def test_gemm_tiled_equals_row_major(case, swiglu, fp8):
    need_gpu()
    cu, rows_cap, k, n, num_w, extra = case
    if swiglu and n % 256:
        n += 128
    a, w, wx = make_inputs(cu, rows_cap, k, n, num_w, extra, seed=len(cu) + k + 7)
    a, w = a.cuda(), w.cuda()
    wx = None if wx is None else wx.cuda()
    kw = {}
    if fp8:
        a, a_s = moe.moe_quantize_act_fp8(a)
        w, w_s = moe.moe_quantize_weight_fp8(w)
        kw = dict(a_scales=a_s, w_scales=w_s)
        if wx is not None:
            wx, wx_s = moe.moe_quantize_weight_fp8(wx)
            kw["w_extra_scales"] = wx_s
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    epi = moe.MOE_EPI_SWIGLU if swiglu else moe.MOE_EPI_NONE
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_r, s_r = moe.moe_grouped_gemm(a, cu_t, w, w_extra=wx, epilogue=epi, dev_status=st, **kw)
    o_t, s_t = moe.moe_grouped_gemm(a, cu_t, moe.moe_pack_weights(w), w_extra=None if wx is None else
                                    moe.moe_pack_weights(wx), epilogue=epi, dev_status=st, tiled=True, **kw)
    torch.cuda.synchronize()
    assert st.item() == 0
    N = cu[-1]
    assert same_bits(o_r[:N], o_t[:N])
    if s_r is not None:
        assert torch.equal(s_r[:N], s_t[:N])


@pytest.mark.parametrize("swiglu,layout,n,n_big,big_rows,k", STREAM_CASES,
                         ids=[f"{'swiglu' if c[0] else 'plain'}-{c[1]}-n{c[2]}" for c in STREAM_CASES])
def test_streaming_launch_tiled_equals_row_major(swiglu, layout, n, n_big, big_rows, k):
    """Launches large enough to run streaming CTAs: the weight stream of the short segments
    and the MMA pipeline both read boxes of the tiled layout (odd N-tile counts, a last
    N-tile half past the weight rows, row_scale, the batched layout)."""
    need_gpu()
    counts = streamed_counts(17 + swiglu + n, n_big, big_rows, 60)
    counts.append(20)
    num_w = len(counts) - 1
    g = torch.Generator().manual_seed(13)
    w = (torch.randn(num_w, n, k, generator=g) / k ** 0.5).to(torch.bfloat16).cuda()
    wx = (torch.randn(n, k, generator=g) / k ** 0.5).to(torch.bfloat16).cuda()
    wt, wxt = moe.moe_pack_weights(w), moe.moe_pack_weights(wx)
    epi = moe.MOE_EPI_SWIGLU if swiglu else moe.MOE_EPI_NONE
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for tiled in (False, True):
        ww, wwx = (wt, wxt) if tiled else (w, wx)
        if layout == "contiguous":
            cu = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).cuda()
            rows = int(sum(counts))
            a = torch.randn(rows, k, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16).cuda()
            rs = None if swiglu else torch.rand(rows, generator=torch.Generator().manual_seed(3)).cuda() + 0.5
            o, _ = moe.moe_grouped_gemm(a, cu, ww, w_extra=wwx, epilogue=epi, dev_status=st, row_scale=rs,
                                        tiled=tiled)
            outs.append(o[:rows])
        else:
            mt = 1024
            S = len(counts)
            a = torch.randn(S, mt, k, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16).cuda()
            rs = None if swiglu else torch.rand(S * mt, generator=torch.Generator().manual_seed(3)).cuda() + 0.5
            o, _ = moe.moe_grouped_gemm_batched(a, torch.tensor(counts, dtype=torch.int32).cuda(), ww, w_extra=wwx,
                                                epilogue=epi, dev_status=st, row_scale=rs, tiled=tiled)
            outs.append(torch.cat([o[s, :counts[s]] for s in range(S)]))
    torch.cuda.synchronize()
    assert st.item() == 0
    assert same_bits(outs[0], outs[1])


LAYER_CASES = [
    # workload, reduced sizes, MoeLayer options
    ("mid", None, {}),
    ("prefill", dict(T=1024, T_valid=768, E=32), {}),
    ("prefill", dict(T=1024, T_valid=768, E=32), dict(weight_in_down=True)),
    ("prefill", dict(T=1024, T_valid=768, E=32), dict(fuse_combine=True)),
    ("prefill", dict(T=512, T_valid=512, E=16), dict(max_tokens=512)),
    ("decode", dict(E=32), {}),
    ("decode", dict(E=32), dict(max_tokens=128)),
]


@pytest.mark.parametrize("name,red,opts", LAYER_CASES,
                         ids=[f"{c[0]}-{'-'.join(c[2]) or 'default'}" for c in LAYER_CASES])
def test_layer_weight_tiles_bit_identical(name, red, opts):
    need_gpu()
    w = WORKLOADS[name] if red is None else scaled(WORKLOADS[name], **red)
    logits = synth.router_logits(w, 0, device="cuda")
    x = synth.hidden(w, 0, device="cuda")
    w13, w2, s13, s2 = synth.expert_weights(w, 0, device="cuda")
    kw = dict(w13=w13, w2=w2, shared_w13=s13, shared_w2=s2)
    dtype = moe.MOE_BF16
    if w.dtype == "e4m3":
        dtype = moe.MOE_E4M3
        q13, c13 = moe.moe_quantize_weight_fp8(w13)
        q2, c2 = moe.moe_quantize_weight_fp8(w2)
        kw = dict(w13=q13, w2=q2, w13_scales=c13, w2_scales=c2)
        if w.shared:
            qs13, cs13 = moe.moe_quantize_weight_fp8(s13)
            qs2, cs2 = moe.moe_quantize_weight_fp8(s2)
            kw.update(shared_w13=qs13, shared_w2=qs2, shared_w13_scales=cs13, shared_w2_scales=cs2)
    if not w.shared:
        kw.update(shared_w13=None, shared_w2=None)
    outs = []
    for tiles in (False, True):
        layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, dtype, weight_tiles=tiles, **opts, **kw)
        idx = torch.empty(w.T, w.K, dtype=torch.int32, device="cuda")
        wt = torch.empty(w.T, w.K, dtype=torch.float32, device="cuda")
        out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        n = torch.tensor([w.T_valid], dtype=torch.int32, device="cuda")
        layer.forward(x, out, idx, wt, logits=logits, num_tokens=n, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_layer_pairs_refuse_tiles():
    need_gpu()
    w = scaled(WORKLOADS["prefill"], T=256, T_valid=256, E=16)
    w13, w2, s13, s2 = synth.expert_weights(w, 0, device="cuda")
    layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, moe.MOE_BF16, w13=w13, w2=w2, shared_w13=s13, shared_w2=s2,
                         gemm_pairs=True, weight_tiles=True)
    with pytest.raises(moe.MoeError) as e:
        layer.forward(synth.hidden(w, 0, device="cuda"), torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda"),
                      torch.empty(w.T, w.K, dtype=torch.int32, device="cuda"),
                      torch.empty(w.T, w.K, dtype=torch.float32, device="cuda"),
                      logits=synth.router_logits(w, 0, device="cuda"))
    assert e.value.code == 3


@pytest.mark.parametrize("swiglu", [False, True])
def test_gemm_tiled_extra_segment_only(swiglu):
    """num_w = 0: the only weights are w_extra (a layer's shared expert alone), tiled."""
    need_gpu()
    k, n = 384, 512
    g = torch.Generator().manual_seed(23)
    a = torch.randn(300, k, generator=g).to(torch.bfloat16).cuda()
    wx = (torch.randn(n, k, generator=g) / k ** 0.5).to(torch.bfloat16).cuda()
    w0 = torch.empty(0, n, k, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 300], dtype=torch.int32, device="cuda")
    epi = moe.MOE_EPI_SWIGLU if swiglu else moe.MOE_EPI_NONE
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_r, _ = moe.moe_grouped_gemm(a, cu, w0, w_extra=wx, epilogue=epi, dev_status=st)
    o_t, _ = moe.moe_grouped_gemm(a, cu, w0, w_extra=moe.moe_pack_weights(wx), epilogue=epi, dev_status=st,
                                  tiled=True)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert same_bits(o_r, o_t)
