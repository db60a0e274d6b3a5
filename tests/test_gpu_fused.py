"""GPU parity of the down projection with the combine fused into its epilogue
(moe_grouped_gemm_combine, the single-GPU part of the Mega-MoE page's one-kernel
GEMM + combine): bit-identical to moe_grouped_gemm + moe_combine and to the oracle's
fixed-order combine of the same rows, in BF16 and E4M3, with and without the shared
expert, router weights, pre-weighted rows, fake-quant, padding tokens, the batched
layout; the counters come back zero so calls repeat; and the layer option
fuse_combine gives the unfused layer's output bit for bit."""
import numpy as np
import pytest
import torch

import combine_moe_route_softmax_gb300 as moe
from combine_moe_route_softmax_gb300 import synth
from combine_moe_route_softmax_gb300.synth import WORKLOADS, scaled
from gpu_helpers import bits, host, need_gpu
from oracle import moe_ref as ref

pytestmark = pytest.mark.gpu


def random_idx(T, K, E, pad, seed, pad_tokens=0):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[rng.random((T, K)) < pad] = -1
    if pad_tokens:
        idx[T - pad_tokens:] = -1        # bucket padding: tokens with no slot at all
    return idx


def problem(T, K, E, I, H, pad, shared, fp8, seed, pad_tokens=0, batched_mt=0):
    idx = random_idx(T, K, E, pad, seed, pad_tokens)
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, I, generator=g).to(torch.bfloat16).cuda()      # stands in for h: the down GEMM input
    dt = moe.MOE_E4M3 if fp8 else moe.MOE_BF16
    if batched_mt:
        lay = moe.moe_permute_batched(torch.from_numpy(idx).cuda(), E, x, batched_mt, with_shared=shared,
                                      out_dtype=dt)
        a, a_s, seg = lay["xb"], lay["xb_scales"], lay["masked_m"]
    else:
        lay = moe.moe_permute(torch.from_numpy(idx).cuda(), E, x, with_shared=shared, out_dtype=dt)
        a, a_s, seg = lay["xp"], lay["xp_scales"], lay["cu_seqlens"]
    w2 = (torch.randn(E, H, I, generator=g) / I ** 0.5).to(torch.bfloat16).cuda()
    ws2 = (torch.randn(H, I, generator=g) / I ** 0.5).to(torch.bfloat16).cuda() if shared else None
    wk = dict(w_extra=ws2)
    if fp8:
        w2, s2 = moe.moe_quantize_weight_fp8(w2)
        wk = dict(w_scales=s2, a_scales=a_s)
        if shared:
            q, sx = moe.moe_quantize_weight_fp8(ws2)
            wk.update(w_extra=q, w_extra_scales=sx)
    wt = torch.rand(T, K, generator=g).cuda()
    return idx, lay, a, seg, w2, wk, wt


CASES = [
    # T, K, E, I, H, slot pad, shared, fp8, pad tokens, batched max_tokens
    (128, 8, 64, 256, 1024, 0.0, True, True, 0, 0),     # decode-shaped, FP8
    (300, 6, 24, 256, 768, 0.15, True, False, 40, 0),   # ragged, bucket padding tokens
    (77, 4, 16, 128, 384, 0.3, False, False, 0, 0),     # no shared expert
    (96, 8, 32, 256, 1024, 0.1, True, True, 10, 96),    # batched layout, FP8
    (64, 2, 8, 256, 256, 0.0, True, False, 0, 64),      # batched, H = 256 (one 256-column tile)
]


@pytest.mark.parametrize("fq", [None, 20.0])
@pytest.mark.parametrize("weighted_rows", [False, True])
@pytest.mark.parametrize("case", CASES, ids=range(len(CASES)))
def test_fused_equals_separate_and_oracle(case, weighted_rows, fq):
    need_gpu()
    T, K, E, I, H, pad, shared, fp8, pad_tokens, mt = case
    idx, lay, a, seg, w2, wk, wt = problem(T, K, E, I, H, pad, shared, fp8, seed=T + H, pad_tokens=pad_tokens,
                                           batched_mt=mt)
    fqt = None if fq is None else torch.tensor([fq], dtype=torch.float32, device="cuda")
    inv, smap, src = lay["inv_map"], lay["shared_map"], lay["src_row"]
    # weighted rows: the permute's per-row weights scale the down GEMM, the combine only sums
    rs = None
    if weighted_rows:
        rw = torch.empty(src.numel(), dtype=torch.float32, device="cuda")
        flat = src.clamp(min=0)
        rw = torch.where(src < T * K, wt.reshape(-1)[flat.clamp(max=T * K - 1)], torch.ones_like(rw))
        rs = rw.contiguous()
    cw = None if weighted_rows else wt
    if mt:
        y_ref, _ = moe.moe_grouped_gemm_batched(a, seg, w2, epilogue=moe.MOE_EPI_NONE, row_scale=rs, **wk)
        y_ref = y_ref.view(-1, H)
    else:
        y_ref, _ = moe.moe_grouped_gemm(a, seg, w2, epilogue=moe.MOE_EPI_NONE, row_scale=rs, **wk)
    out_ref = moe.moe_combine(y_ref, inv, cw, shared_y=y_ref if shared else None, shared_map=smap, fq_scale=fqt)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sentinel = torch.full((T, H), 0x7FC1, dtype=torch.int16).view(torch.bfloat16).cuda()
    out, y, cnt = moe.moe_grouped_gemm_combine(a, seg, w2, src, inv, cw, max_tokens=mt, shared_map=smap,
                                               fq_scale=fqt, row_scale=rs, out=sentinel, dev_status=st, **wk)
    torch.cuda.synchronize()
    assert st.item() == 0
    # the expert rows that exist, the combined output and the oracle's combine of those rows
    rows = host(src) >= 0
    assert np.array_equal(bits(y)[rows], bits(y_ref)[rows])
    assert np.array_equal(bits(out), bits(out_ref))
    yb = bits(y)
    want = ref.combine(yb, host(inv), None if cw is None else host(cw), shared_bits=yb if shared else None,
                       shared_map=None if smap is None else host(smap), fq_scale=fq)
    assert np.array_equal(bits(out), want)
    if pad_tokens:
        assert np.all(bits(out)[T - pad_tokens:] == 0)
    assert not torch.any(cnt)                # counters back to zero
    # a second call on the same counters gives the same result
    out2, _, cnt2 = moe.moe_grouped_gemm_combine(a, seg, w2, src, inv, cw, max_tokens=mt, shared_map=smap,
                                                 fq_scale=fqt, row_scale=rs, counters=cnt, **wk)
    assert np.array_equal(bits(out2), bits(out)) and not torch.any(cnt2)


def test_fused_all_padding_batch_writes_zeros():
    need_gpu()
    T, K, E, I, H = 50, 4, 8, 128, 256
    idx = np.full((T, K), -1, np.int32)
    x = torch.randn(T, I).to(torch.bfloat16).cuda()
    lay = moe.moe_permute(torch.from_numpy(idx).cuda(), E, x, with_shared=True)
    w2 = torch.randn(E, H, I).to(torch.bfloat16).cuda()
    out = torch.full((T, H), 0x7FC1, dtype=torch.int16).view(torch.bfloat16).cuda()
    moe.moe_grouped_gemm_combine(lay["xp"], lay["cu_seqlens"], w2, lay["src_row"], lay["inv_map"],
                                 torch.rand(T, K).cuda(), shared_map=lay["shared_map"],
                                 w_extra=torch.randn(H, I).to(torch.bfloat16).cuda(), out=out)
    torch.cuda.synchronize()
    assert np.all(bits(out) == 0)


def layer_out(w, fuse, max_tokens=0, weight_in_down=False, fq=None, seed=0):
    logits = synth.router_logits(w, seed, device="cuda")
    x = synth.hidden(w, seed, device="cuda")
    w13, w2, s13, s2 = synth.expert_weights(w, seed, device="cuda")
    kw = dict(w13=w13, w2=w2, shared_w13=s13, shared_w2=s2)
    dt = moe.MOE_BF16
    if w.dtype == "e4m3":
        q13, c13 = moe.moe_quantize_weight_fp8(w13)
        q2, c2 = moe.moe_quantize_weight_fp8(w2)
        kw = dict(w13=q13, w2=q2, w13_scales=c13, w2_scales=c2)
        if s13 is not None:
            a, b = moe.moe_quantize_weight_fp8(s13)
            c, d = moe.moe_quantize_weight_fp8(s2)
            kw.update(shared_w13=a, shared_w13_scales=b, shared_w2=c, shared_w2_scales=d)
        dt = moe.MOE_E4M3
    layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, dt, weight_in_down=weight_in_down, max_tokens=max_tokens,
                         fuse_combine=fuse, **kw)
    layer.ws.fill_(0x5A)                      # the layer must not rely on a zeroed workspace
    idx = torch.empty(w.T, w.K, dtype=torch.int32, device="cuda")
    wt = torch.empty(w.T, w.K, dtype=torch.float32, device="cuda")
    out = torch.full((w.T, w.H), 0x7FC1, dtype=torch.int16).view(torch.bfloat16).cuda()
    n = torch.tensor([w.T_valid], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fqt = None if fq is None else torch.tensor([fq], dtype=torch.float32, device="cuda")
    for _ in range(2):                        # twice: the second call starts from the counters the first left
        layer.forward(x, out, idx, wt, logits=logits, num_tokens=n, fq_scale=fqt, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return bits(out)


@pytest.mark.parametrize("case", ["tiny", "decode_fp8", "prefill_small_fq", "prefill_small_wd", "decode_batched",
                                  "decode_full"])
def test_layer_fused_combine_equals_unfused(case):
    need_gpu()
    kw = {}
    if case == "tiny":
        w = WORKLOADS["tiny"]
    elif case == "decode_fp8":
        w = scaled(WORKLOADS["decode"], H=1024, I=512, E=64)
    elif case == "prefill_small_fq":
        w = scaled(WORKLOADS["prefill"], T=256, T_valid=200, H=768, I=256, E=16, K=4)
        kw = dict(fq=25.0)
    elif case == "prefill_small_wd":
        w = scaled(WORKLOADS["prefill"], T=256, T_valid=200, H=768, I=256, E=16, K=4)
        kw = dict(weight_in_down=True)
    elif case == "decode_batched":
        w = scaled(WORKLOADS["decode"], H=1024, I=512, E=64)
        kw = dict(max_tokens=128)
    else:
        w = WORKLOADS["decode"]
    a = layer_out(w, False, **kw)
    b = layer_out(w, True, **kw)
    assert np.array_equal(a, b)
