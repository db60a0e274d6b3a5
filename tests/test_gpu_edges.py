"""GPU edge cases of the whole layer and the grouped GEMM: degenerate sizes, an all-padding
batch, expert ids out of range, the largest segment count, and an FP8 layer replayed from a
CUDA graph -- each against the oracle or against an eager run."""
import numpy as np
import pytest
import torch

import combine_moe_route_softmax_gb300 as moe
from combine_moe_route_softmax_gb300 import synth
from combine_moe_route_softmax_gb300.synth import WORKLOADS, scaled
from gpu_helpers import ExpertBits, bits, host, need_gpu
from oracle import moe_ref as ref
from oracle.formats import bf16_bits_to_f32

pytestmark = pytest.mark.gpu


def make_layer(w, seed=0, fp8=False):
    x = synth.hidden(w, seed, device="cuda")
    logits = synth.router_logits(w, seed, device="cuda")
    w13, w2, s13, s2 = synth.expert_weights(w, seed, device="cuda")
    kw = dict(w13=w13, w2=w2, shared_w13=s13, shared_w2=s2)
    if fp8:
        q13, c13 = moe.moe_quantize_weight_fp8(w13)
        q2, c2 = moe.moe_quantize_weight_fp8(w2)
        kw = dict(w13=q13, w2=q2, w13_scales=c13, w2_scales=c2)
        if w.shared:
            a, b = moe.moe_quantize_weight_fp8(s13)
            c, d = moe.moe_quantize_weight_fp8(s2)
            kw.update(shared_w13=a, shared_w13_scales=b, shared_w2=c, shared_w2_scales=d)
    layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, moe.MOE_E4M3 if fp8 else moe.MOE_BF16, **kw)
    bufs = dict(idx=torch.empty(w.T, w.K, dtype=torch.int32, device="cuda"),
                wt=torch.empty(w.T, w.K, dtype=torch.float32, device="cuda"),
                out=torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda"),
                n=torch.tensor([w.T_valid], dtype=torch.int32, device="cuda"),
                st=torch.zeros(1, dtype=torch.int32, device="cuda"))
    return x, logits, (w13, w2, s13, s2), layer, bufs


@pytest.mark.parametrize("T,H,I,E,K,shared", [(1, 128, 128, 1, 1, False), (1, 256, 128, 4, 2, True),
                                              (13, 384, 256, 3, 3, True), (200, 128, 384, 200, 1, False),
                                              # top-k above 8: the 32-slot combine, wide permute scatter
                                              (50, 256, 256, 64, 16, True), (20, 128, 128, 40, 32, False)])
def test_degenerate_layers(T, H, I, E, K, shared):
    need_gpu()
    w = scaled(WORKLOADS["tiny"], T=T, T_valid=T, H=H, I=I, E=E, K=K, shared=shared)
    x, logits, (w13, w2, s13, s2), layer, b = make_layer(w)
    layer.forward(x, b["out"], b["idx"], b["wt"], logits=logits, num_tokens=b["n"], dev_status=b["st"])
    torch.cuda.synchronize()
    assert b["st"].item() == 0
    o_idx, o_w = ref.route_topk(host(logits), K)
    assert np.array_equal(host(b["idx"]), o_idx)
    want = ref.layer_reference(bits(x), o_idx, o_w, ExpertBits(w13), ExpertBits(w2),
                               shared=(bits(s13), bits(s2)) if shared else None)
    err = ref.max_rel_err(bf16_bits_to_f32(bits(b["out"])).astype(np.float64), want)
    assert err <= 2e-2, err


def test_all_padding_batch_gives_zeros():
    need_gpu()
    w = scaled(WORKLOADS["prefill"], T=64, T_valid=0, H=256, I=128, E=8, K=2)
    x, logits, _, layer, b = make_layer(w)
    b["out"].fill_(1.0)
    layer.forward(x, b["out"], b["idx"], b["wt"], logits=logits, num_tokens=b["n"], dev_status=b["st"])
    torch.cuda.synchronize()
    assert b["st"].item() == 0
    assert np.all(host(b["idx"]) == -1)
    assert np.all(bits(b["out"]) == 0)
    cu = host(layer.view("cu_seqlens", (w.E + 2,), torch.int32))
    assert np.all(cu == 0)


def test_out_of_range_ids_are_flagged_and_skipped():
    need_gpu()
    w = scaled(WORKLOADS["tiny"], T=32, T_valid=32, H=256, I=128, E=8, K=2, shared=True)
    x, logits, (w13, w2, s13, s2), layer, b = make_layer(w)
    o_idx, o_w = ref.route_topk(host(logits), w.K)
    bad = o_idx.copy()
    bad[3, 1] = 8          # == E
    bad[7, 0] = 1000
    bad[9, 1] = -5
    b["idx"].copy_(torch.from_numpy(bad))
    b["wt"].copy_(torch.from_numpy(o_w))
    layer.forward(x, b["out"], b["idx"], b["wt"], dev_status=b["st"])
    torch.cuda.synchronize()
    assert b["st"].item() & moe.MOE_DEV_BAD_EXPERT
    skipped = np.where((bad >= 0) & (bad < w.E), bad, -1).astype(np.int32)
    want = ref.layer_reference(bits(x), skipped, o_w, ExpertBits(w13), ExpertBits(w2), shared=(bits(s13), bits(s2)))
    err = ref.max_rel_err(bf16_bits_to_f32(bits(b["out"])).astype(np.float64), want)
    assert err <= 2e-2, err


def test_gemm_with_the_largest_segment_count():
    need_gpu()
    E = 1024                                  # + one extra segment = 1025 segments
    rng = np.random.default_rng(3)
    counts = rng.integers(0, 4, E + 1)
    counts[::97] = 130                        # a few multi-tile segments
    cu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows, k, n = int(cu[-1]), 128, 256
    g = torch.Generator().manual_seed(4)
    a = torch.randn(rows, k, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, n, k, generator=g) / k ** 0.5).to(torch.bfloat16)
    wx = (torch.randn(n, k, generator=g) / k ** 0.5).to(torch.bfloat16)
    out, _ = moe.moe_grouped_gemm(a.cuda(), torch.from_numpy(cu).cuda(), w.cuda(), w_extra=wx.cuda())
    f = lambda t: bf16_bits_to_f32(bits(t)).astype(np.float64)
    a64, w64, wx64 = f(a), f(w), f(wx)
    want = np.concatenate([a64[cu[s]:cu[s + 1]] @ (w64[s] if s < E else wx64).T for s in range(E + 1)])
    got = f(out)
    scale = np.abs(want).max()
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 2e-3 * scale)


def test_fp8_layer_replayed_from_a_cuda_graph():
    need_gpu()
    w = scaled(WORKLOADS["decode"], T=64, T_valid=64, H=1024, I=512, E=16, K=4)
    x, logits, _, layer, b = make_layer(w, fp8=True)
    run = lambda: layer.forward(x, b["out"], b["idx"], b["wt"], logits=logits, num_tokens=b["n"],
                                dev_status=b["st"])
    run()
    torch.cuda.synchronize()
    eager = bits(b["out"]).copy()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    b["out"].zero_()
    g.replay()
    torch.cuda.synchronize()
    assert b["st"].item() == 0
    assert np.array_equal(bits(b["out"]), eager)


def test_one_graph_replayed_at_every_bucket_fill():
    """A layer captured once serves batches of any fill of its bucket: num_tokens is read on
    the device, so each replay routes, permutes and combines only the first n rows (the
    rest come out +0), bit-identical to an eager call with the same n."""
    need_gpu()
    w = scaled(WORKLOADS["prefill"], T=256, T_valid=256, H=512, I=256, E=16, K=4)
    x, logits, _, layer, b = make_layer(w)
    run = lambda: layer.forward(x, b["out"], b["idx"], b["wt"], logits=logits, num_tokens=b["n"],
                                dev_status=b["st"])
    run()                                       # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for n in (256, 0, 1, 37, 200, 256):
        b["n"].fill_(n)
        b["out"].fill_(7.0)
        run()
        torch.cuda.synchronize()
        eager = bits(b["out"]).copy()
        b["out"].fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        assert b["st"].item() == 0
        assert np.array_equal(bits(b["out"]), eager), n
        assert np.all(eager[n:] == 0) and np.all(host(b["idx"])[n:] == -1)


def test_fp8_layer_with_twelve_experts_per_token():
    """E4M3 layer with K = 12 and a shared expert against the oracle on the FP8 operands."""
    need_gpu()
    w = scaled(WORKLOADS["decode"], T=48, T_valid=48, H=512, I=256, E=32, K=12)
    x, logits, (w13, w2, s13, s2), layer, b = make_layer(w, fp8=True)
    layer.forward(x, b["out"], b["idx"], b["wt"], logits=logits, num_tokens=b["n"], dev_status=b["st"])
    torch.cuda.synchronize()
    assert b["st"].item() == 0
    o_idx, o_w = ref.route_topk(host(logits), w.K)
    assert np.array_equal(host(b["idx"]), o_idx)
    want = ref.layer_reference(bits(x), o_idx, o_w, ExpertBits(w13), ExpertBits(w2), shared=(bits(s13), bits(s2)),
                               fp8=True)
    err = ref.max_rel_err(bf16_bits_to_f32(bits(b["out"])).astype(np.float64), want)
    assert err <= 6e-2, err
