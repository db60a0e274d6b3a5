"""GPU parity of the NVFP4 combine fake-quant (two-level NVFP4 reading: 16-column blocks,
E4M3 block scales, per-tensor scale 448*6/amax, E2M1 elements): bit-exact against the
oracle's combine on the same BF16 rows (padding slots, shared rows, pre-weighted rows,
the split-column path for few tokens, K > 8), the per-tensor scale, the on-grid identity,
and the layer option, whose output the oracle re-sums from the layer's own expert rows."""
import numpy as np
import pytest
import torch

import combine_moe_route_softmax_gb300 as moe
from combine_moe_route_softmax_gb300 import synth
from combine_moe_route_softmax_gb300.synth import WORKLOADS, scaled
from gpu_helpers import bits, host, need_gpu
from oracle import moe_ref as ref
from oracle.formats import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def combine_problem(T, K, E, H, pad, shared, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[rng.random((T, K)) < pad] = -1
    cu, src, inv, smap, _ = ref.permute(idx, E, with_shared=shared)
    g = torch.Generator("cuda").manual_seed(seed)
    # rows with per-row magnitudes spread over four decades, so block scales vary
    y = (torch.randn(len(src), H, generator=g, device="cuda") *
         torch.exp(torch.randn(len(src), 1, generator=g, device="cuda") * 2)).to(torch.bfloat16)
    wt = torch.rand(T, K, generator=g, device="cuda")
    return inv, smap, y, wt


@pytest.mark.parametrize("T,K,E,H,pad,shared,weighted", [
    (333, 8, 64, 1024, 0.1, True, False),
    (50, 2, 8, 256, 0.0, False, False),
    (64, 12, 16, 384, 0.2, True, False),       # K > 8
    (200, 4, 16, 512, 0.25, False, True),      # rows already router-weighted (topk_w NULL)
    (1, 8, 64, 7168, 0.0, True, False),        # few tokens: columns split over warps
    (5, 8, 64, 7168, 0.1, True, False),
    (7, 4, 9, 1152, 0.2, False, False),        # 144 vectors: split parts rounded to whole blocks
    (1024, 8, 256, 7168, 0.0, True, False),
])
def test_combine_nvfp4_bit_exact(T, K, E, H, pad, shared, weighted):
    need_gpu()
    inv, smap, y, wt = combine_problem(T, K, E, H, pad, shared, seed=T + K + H)
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    invd = torch.from_numpy(inv).cuda()
    moe.moe_combine_amax(y, invd, None if weighted else wt, amax)
    g = moe.moe_fq4_scale_from_amax(amax)
    oa = ref.combine_amax(bits(y), inv, None if weighted else host(wt))
    assert host(amax)[0] == oa and host(g)[0] == ref.nvfp4_scale_from_amax(oa)
    # a scale 4x above the calibrated one as well: saturated block scales and elements
    for gs in (host(g)[0], np.float32(host(g)[0] * 4)):
        gt = torch.tensor([gs], dtype=torch.float32, device="cuda")
        out = moe.moe_combine_nvfp4(y, invd, None if weighted else wt, gt, shared_y=y if shared else None,
                                    shared_map=torch.from_numpy(smap).cuda() if shared else None)
        yb = bits(y)
        want = ref.combine(yb, inv, None if weighted else host(wt), shared_bits=yb if shared else None,
                           shared_map=smap, fq_scale=gs, fq_format="nvfp4")
        assert np.array_equal(bits(out), want)


def test_combine_nvfp4_on_grid_rows_is_the_plain_combine():
    """Rows of E2M1 values times a power of two per 16-column block (one element at 6 per
    block), weights 1, g = 1: the fake-quant returns every row unchanged."""
    need_gpu()
    rng = np.random.default_rng(8)
    T, K, H = 40, 4, 256
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    v = rng.choice(grid, size=(T * K, H // 16, 16)) * rng.choice([-1.0, 1.0], size=(T * K, H // 16, 16))
    v[:, :, 0] = 6.0
    v = v * np.exp2(rng.integers(-6, 6, size=(T * K, H // 16, 1)))
    y = torch.from_numpy(f32_to_bf16_bits(v.reshape(T * K, H).astype(np.float32)).view(np.int16)).view(
        torch.bfloat16).cuda()
    inv = torch.arange(T * K, dtype=torch.int32, device="cuda").reshape(T, K)
    w = torch.ones(T, K, device="cuda")
    g = torch.ones(1, device="cuda")
    assert np.array_equal(bits(moe.moe_combine_nvfp4(y, inv, w, g)), bits(moe.moe_combine(y, inv, w)))


def test_layer_with_nvfp4_combine():
    need_gpu()
    w = scaled(WORKLOADS["prefill"], T=96, T_valid=72, H=512, I=256, E=16, K=4)
    x = synth.hidden(w, 0, device="cuda")
    logits = synth.router_logits(w, 0, device="cuda")
    w13, w2, s13, s2 = synth.expert_weights(w, 0, device="cuda")
    layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, moe.MOE_BF16, w13=w13, w2=w2, shared_w13=s13, shared_w2=s2,
                         combine_fq="nvfp4")
    idx = torch.empty(w.T, w.K, dtype=torch.int32, device="cuda")
    wt = torch.empty(w.T, w.K, dtype=torch.float32, device="cuda")
    out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    n = torch.tensor([w.T_valid], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # calibrate on the batch itself: the layer once without fake-quant, then the amax
    layer.forward(x, out, idx, wt, logits=logits, num_tokens=n, dev_status=st)
    v, d = layer.views, layer.desc
    y = layer.view("y", (v.cap, d.H), torch.bfloat16)
    inv = layer.view("inv_map", (d.T, d.K), torch.int32)
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    moe.moe_combine_amax(y, inv, wt, amax)
    g = moe.moe_fq4_scale_from_amax(amax)
    plain = bits(out).copy()
    layer.forward(x, out, idx, wt, logits=logits, num_tokens=n, fq_scale=g, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    smap = host(layer.view("shared_map", (d.T,), torch.int32))
    yb = bits(y)
    want = ref.combine(yb, host(inv), host(wt), shared_bits=yb, shared_map=smap, fq_scale=host(g)[0],
                       fq_format="nvfp4")
    assert np.array_equal(bits(out), want)
    assert not np.array_equal(bits(out), plain)
    assert np.all(bits(out)[w.T_valid:] == 0)


def test_nvfp4_combine_with_the_fused_combine_is_rejected():
    need_gpu()
    w = scaled(WORKLOADS["tiny"], T=16, T_valid=16, H=256, I=128, E=4, K=2)
    w13, w2, _, _ = synth.expert_weights(w, 0, device="cuda")
    layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, moe.MOE_BF16, w13=w13, w2=w2, fuse_combine=True, combine_fq="nvfp4")
    x = synth.hidden(w, 0, device="cuda")
    logits = synth.router_logits(w, 0, device="cuda")
    out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(w.T, w.K, dtype=torch.int32, device="cuda")
    wt = torch.empty(w.T, w.K, dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        layer.forward(x, out, idx, wt, logits=logits, fq_scale=torch.ones(1, device="cuda"))
    assert e.value.code == 3


def test_combine_nvfp4_rounds_exact_ties_to_even_codes():
    """Blocks whose scaled elements sit exactly on E2M1 midpoints (0.25, 0.75, ..., 5) and
    beyond the largest value: each tie goes to the even code, as the oracle's E2M1."""
    need_gpu()
    T, K, H = 8, 2, 128
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0])
    rows = np.zeros((T * K, H // 16, 16))
    rows[:, :, 0] = 6.0                                     # block amax 6: scale 1 at g = 1
    rows[:, :, 1:] = ties
    rows = rows * np.exp2(np.arange(T * K) % 5 - 2)[:, None, None]
    y = torch.from_numpy(f32_to_bf16_bits(rows.reshape(T * K, H).astype(np.float32)).view(np.int16)).view(
        torch.bfloat16).cuda()
    inv = np.arange(T * K, dtype=np.int32).reshape(T, K)
    w = np.ones((T, K), dtype=np.float32)
    g = np.float32(1.0)
    out = moe.moe_combine_nvfp4(y, torch.from_numpy(inv).cuda(), torch.from_numpy(w).cuda(),
                                torch.tensor([g], device="cuda"))
    want = ref.combine(bits(y), inv, w, fq_scale=g, fq_format="nvfp4")
    assert np.array_equal(bits(out), want)
    # and the ties did move: the fake-quantised sum differs from the plain one
    assert not np.array_equal(want, ref.combine(bits(y), inv, w))


@pytest.mark.parametrize("T,K,E,H,shared,layout", [
    (300, 8, 64, 1024, True, "contiguous"),
    (3, 8, 64, 7168, True, "contiguous"),      # few tokens: columns split over warps
    (40, 4, 16, 1152, False, "contiguous"),    # 144 vectors: a ragged last group
    (64, 4, 16, 512, True, "batched"),
])
def test_permute_nvfp4_dispatch_bit_exact(T, K, E, H, shared, layout):
    """Routed rows get the NVFP4 fake-quant of x (BF16 result), shared rows the original."""
    need_gpu()
    rng = np.random.default_rng(T + H)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    g0 = torch.Generator("cuda").manual_seed(T)
    x = (torch.randn(T, H, generator=g0, device="cuda") *
         torch.exp(torch.randn(T, 1, generator=g0, device="cuda"))).to(torch.bfloat16)
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    moe.moe_amax_bf16(x, amax)
    g = moe.moe_fq4_scale_from_amax(amax)
    gs = host(g)[0]
    assert gs == ref.nvfp4_scale_from_amax(ref.tensor_amax(bits(x)))
    idx_d = torch.from_numpy(idx).cuda()
    if layout == "contiguous":
        res = moe.moe_permute(idx_d, E, x, with_shared=shared, dispatch_scale=g, dispatch_format="nvfp4")
        rows_out = bits(res["xp"])
        src = host(res["src_row"])
    else:
        res = moe.moe_permute_batched(idx_d, E, x, T, with_shared=shared, dispatch_scale=g, dispatch_format="nvfp4")
        rows_out = bits(res["xb"]).reshape(-1, H)
        src = host(res["src_row"])
    xq = ref.dispatch_qdq_bits(bits(x), gs, "nvfp4")
    xb = bits(x)
    TK = T * K
    for r, sidx in enumerate(src):
        if sidx < 0:
            continue
        if sidx < TK:
            assert np.array_equal(rows_out[r], xq[sidx // K]), r
        else:
            assert np.array_equal(rows_out[r], xb[sidx - TK]), r


def test_layer_with_nvfp4_dispatch():
    need_gpu()
    w = scaled(WORKLOADS["prefill"], T=96, T_valid=72, H=512, I=256, E=16, K=4)
    x = synth.hidden(w, 0, device="cuda")
    logits = synth.router_logits(w, 0, device="cuda")
    w13, w2, s13, s2 = synth.expert_weights(w, 0, device="cuda")
    layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, moe.MOE_BF16, w13=w13, w2=w2, shared_w13=s13, shared_w2=s2,
                         dispatch_fq="nvfp4")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    moe.moe_amax_bf16(x[:w.T_valid], amax)
    g = moe.moe_fq4_scale_from_amax(amax)
    idx = torch.empty(w.T, w.K, dtype=torch.int32, device="cuda")
    wt = torch.empty(w.T, w.K, dtype=torch.float32, device="cuda")
    out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    n = torch.tensor([w.T_valid], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer.forward(x, out, idx, wt, logits=logits, num_tokens=n, dispatch_scale=g, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    from gpu_helpers import ExpertBits
    from oracle.formats import bf16_bits_to_f32
    want = ref.layer_reference(bits(x), host(idx), host(wt), ExpertBits(w13), ExpertBits(w2),
                               shared=(bits(s13), bits(s2)), tokens=np.arange(w.T_valid),
                               dispatch_scale=host(g)[0], dispatch_format="nvfp4")
    got = bf16_bits_to_f32(bits(out)).astype(np.float64)[:w.T_valid]
    assert ref.max_rel_err(got, want) <= 2e-2
    # the format matters: the E4M3 reading of the same scale gives another output
    plain = ref.layer_reference(bits(x), host(idx), host(wt), ExpertBits(w13), ExpertBits(w2),
                                shared=(bits(s13), bits(s2)), tokens=np.arange(w.T_valid))
    assert ref.max_rel_err(got, plain) > 5e-3


def test_layer_with_every_option_together():
    """NVFP4 dispatch and combine, router weights in the down projection and the batched
    layout in one layer: the output is the oracle's NVFP4 re-sum of the layer's own
    (weighted) expert rows, bit for bit, and the routed input rows are the oracle's NVFP4
    dispatch of x."""
    need_gpu()
    w = scaled(WORKLOADS["prefill"], T=64, T_valid=48, H=512, I=256, E=8, K=4)
    x = synth.hidden(w, 0, device="cuda")
    logits = synth.router_logits(w, 0, device="cuda")
    w13, w2, s13, s2 = synth.expert_weights(w, 0, device="cuda")
    layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, moe.MOE_BF16, w13=w13, w2=w2, shared_w13=s13, shared_w2=s2,
                         weight_in_down=True, max_tokens=w.T, combine_fq="nvfp4", dispatch_fq="nvfp4")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    moe.moe_amax_bf16(x[:w.T_valid], amax)
    gd = moe.moe_fq4_scale_from_amax(amax)
    gc = torch.tensor([200.0], dtype=torch.float32, device="cuda")
    idx = torch.empty(w.T, w.K, dtype=torch.int32, device="cuda")
    wt = torch.empty(w.T, w.K, dtype=torch.float32, device="cuda")
    out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    n = torch.tensor([w.T_valid], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer.forward(x, out, idx, wt, logits=logits, num_tokens=n, fq_scale=gc, dispatch_scale=gd, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    v, d = layer.views, layer.desc
    y = layer.view("y", (v.cap, d.H), torch.bfloat16)
    xp = layer.view("xp", (v.cap, d.H), torch.bfloat16)
    inv = host(layer.view("inv_map", (d.T, d.K), torch.int32))
    src = host(layer.view("src_row", (v.cap,), torch.int32))
    smap = host(layer.view("shared_map", (d.T,), torch.int32))
    yb = bits(y)
    # rows are stored weighted: the combine only sums (topk_w None)
    want = ref.combine(yb, inv, None, shared_bits=yb, shared_map=smap, fq_scale=np.float32(200.0), fq_format="nvfp4")
    assert np.array_equal(bits(out), want)
    xq = ref.dispatch_qdq_bits(bits(x), host(gd)[0], "nvfp4")
    xpb = bits(xp)
    TK = w.T * w.K
    checked = 0
    for r, s_ in enumerate(src):
        if s_ < 0:
            continue
        assert np.array_equal(xpb[r], xq[s_ // w.K] if s_ < TK else bits(x)[s_ - TK]), r
        checked += 1
    assert checked == int((inv >= 0).sum()) + int((smap >= 0).sum())
