"""GPU parity of the expert-batched layout ([E, max_tokens, H] with per-expert row counts,
the DeepEP page's low-latency format) against the oracle: moe_permute_batched bit-exact
(every index array, every kept row, BF16 and E4M3, with overflow), moe_grouped_gemm_batched
against fp64 per-block products (ragged masked_m, out-of-range counts clamped, untouched
padding rows), and the whole layer in the batched layout: bit-identical to the contiguous
layout (each output row depends only on its own input row) and within tolerance of the
oracle."""
import numpy as np
import pytest
import torch

import combine_moe_route_softmax_gb300 as moe
from combine_moe_route_softmax_gb300 import synth
from combine_moe_route_softmax_gb300.synth import WORKLOADS, scaled
from gpu_helpers import ExpertBits, bits, host, need_gpu
from oracle import moe_ref as ref
from oracle.formats import bf16_bits_to_f32, e4m3_decode

pytestmark = pytest.mark.gpu

SENTINEL = 0x7FC1


def random_idx(T, K, E, pad, seed, skew=0):
    rng = np.random.default_rng(seed)
    p = np.ones(E)
    p[:4] += skew
    idx = np.stack([rng.choice(E, K, replace=False, p=p / p.sum()) for _ in range(T)]).astype(np.int32)
    idx[rng.random((T, K)) < pad] = -1
    return idx


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("mt", [37, 400])
def test_permute_batched_bit_exact(mt, shared, fp8):
    need_gpu()
    T, K, E, H = 300, 6, 24, 512
    idx = random_idx(T, K, E, 0.15, seed=3, skew=6)   # skewed: the first experts overflow at 37
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = moe.moe_permute_batched(torch.from_numpy(idx).cuda(), E, x.cuda(), mt, with_shared=shared,
                                  out_dtype=moe.MOE_E4M3 if fp8 else moe.MOE_BF16, dev_status=st)
    torch.cuda.synchronize()
    m, src, inv, smap, ost = ref.permute_batched(idx, E, mt, with_shared=shared)
    assert np.array_equal(host(res["masked_m"]), m)
    assert np.array_equal(host(res["src_row"]), src)
    assert np.array_equal(host(res["inv_map"]), inv)
    if shared:
        assert np.array_equal(host(res["shared_map"]), smap)
    assert st.item() == ost and (ost == ref.STATUS_OVERFLOW) == (mt == 37)
    rows = np.nonzero(src >= 0)[0]
    tok = ref.row_tokens(src[rows], T, K)
    if fp8:
        q, s = ref.act_quant_1x128(bf16_bits_to_f32(bits(x)))
        nseg = E + int(shared)
        assert np.array_equal(host(res["xb"]).reshape(nseg * mt, H)[rows], q[tok])
        assert np.array_equal(host(res["xb_scales"]).reshape(nseg * mt, -1)[rows], s[tok])
    else:
        assert np.array_equal(bits(res["xb"]).reshape(-1, H)[rows], bits(x)[tok])


def test_permute_batched_decode_workload():
    need_gpu()
    w = WORKLOADS["decode"]
    logits = synth.router_logits(w, 0, device="cuda")
    idx, _ = moe.moe_route_topk(logits, w.K)
    x = synth.hidden(w, 0, device="cuda")
    res = moe.moe_permute_batched(idx, w.E, x, w.T, with_shared=True, out_dtype=moe.MOE_E4M3)
    m, src, inv, smap, st = ref.permute_batched(host(idx), w.E, w.T, with_shared=True)
    assert st == 0
    for k, v in (("masked_m", m), ("src_row", src), ("inv_map", inv), ("shared_map", smap)):
        assert np.array_equal(host(res[k]), v), k


def test_permute_batched_empty_batch():
    need_gpu()
    idx = torch.zeros(0, 4, dtype=torch.int32, device="cuda")
    x = torch.zeros(0, 256, dtype=torch.bfloat16, device="cuda")
    res = moe.moe_permute_batched(idx, 8, x, 16, with_shared=True)
    torch.cuda.synchronize()
    assert np.all(host(res["masked_m"]) == 0) and np.all(host(res["src_row"]) == -1)


def gemm_reference(a64, wl, m, mt, swiglu):
    out = {}
    for s, n in enumerate(m):
        acc = a64[s * mt:s * mt + n] @ wl[s].T
        if swiglu:
            I = acc.shape[1] // 2
            g, u = acc[:, :I], acc[:, I:]
            with np.errstate(over="ignore"):
                acc = g / (1.0 + np.exp(-g)) * u
        out[s] = acc
    return out


@pytest.mark.parametrize("swiglu", [False, True])
@pytest.mark.parametrize("fp8", [False, True])
def test_grouped_gemm_batched(fp8, swiglu):
    need_gpu()
    mt, k, n, num_w = 200, 256, 512, 5
    masked = [0, 1, 250, 77, -3, 130]       # 250 clamps to 200, -3 to 0; segment 5 uses w_extra
    m = [min(max(v, 0), mt) for v in masked]
    S = len(masked)
    g = torch.Generator().manual_seed(5)
    a = torch.randn(S * mt, k, generator=g).to(torch.bfloat16)
    w = (torch.randn(num_w, n, k, generator=g) / k ** 0.5).to(torch.bfloat16)
    wx = (torch.randn(n, k, generator=g) / k ** 0.5).to(torch.bfloat16)
    mm = torch.tensor(masked, dtype=torch.int32, device="cuda")
    cols = n // 2 if swiglu else n
    epi = moe.MOE_EPI_SWIGLU if swiglu else moe.MOE_EPI_NONE
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    T_ = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()
    if fp8:
        qa, sa = ref.act_quant_1x128(bf16_bits_to_f32(bits(a)))
        qw, sw = zip(*[ref.weight_quant_128x128(bf16_bits_to_f32(bits(w[i]))) for i in range(num_w)])
        qx, sx = ref.weight_quant_128x128(bf16_bits_to_f32(bits(wx)))
        a64 = ref.dequant(qa, sa, 1)
        wl = [ref.dequant(qw[s], sw[s], 128) for s in range(num_w)] + [ref.dequant(qx, sx, 128)]
        if swiglu:
            out = torch.zeros(S, mt, cols, dtype=torch.uint8, device="cuda")
            out_s = torch.full((S, mt, cols // 128), -1.0, dtype=torch.float32, device="cuda")
        else:
            out = torch.full((S, mt, cols), SENTINEL, dtype=torch.int16).view(torch.bfloat16).cuda()
            out_s = None
        moe.moe_grouped_gemm_batched(T_(qa).view(S, mt, k), mm, T_(np.stack(qw)), a_scales=T_(sa),
                                     w_scales=T_(np.stack(sw)), w_extra=T_(qx), w_extra_scales=T_(sx), epilogue=epi,
                                     out=out, out_scales=out_s, dev_status=st)
    else:
        f = lambda t: bf16_bits_to_f32(bits(t)).astype(np.float64)
        a64, wl = f(a), [f(w[s]) for s in range(num_w)] + [f(wx)]
        out = torch.full((S, mt, cols), SENTINEL, dtype=torch.int16).view(torch.bfloat16).cuda()
        out_s = None
        moe.moe_grouped_gemm_batched(a.cuda().view(S, mt, k), mm, w.cuda(), w_extra=wx.cuda(), epilogue=epi,
                                     out=out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    want = gemm_reference(a64, wl, m, mt, swiglu)
    for s in range(S):
        if fp8 and swiglu:
            gq, gs = host(out)[s], host(out_s)[s]
            if m[s]:
                got = e4m3_decode(gq[:m[s]]).astype(np.float64) * np.repeat(gs[:m[s]].astype(np.float64), 128, 1)
                scale = np.abs(want[s]).max()
                srep = np.repeat(gs[:m[s]].astype(np.float64), 128, axis=1)
                assert np.all(np.abs(got - want[s]) <= 2.0 ** -4 * np.abs(want[s]) * 1.01 + srep * 2.0 ** -9
                              + 1e-3 * scale)
            assert np.all(gs[m[s]:] == -1.0)       # padding rows of the block untouched
        else:
            ob = bits(out[s])
            if m[s]:
                got = bf16_bits_to_f32(ob[:m[s]]).astype(np.float64)
                scale = np.abs(want[s]).max()
                assert np.all(np.abs(got - want[s]) <= 2.0 ** -8 * np.abs(want[s]) + 2e-3 * scale)
            assert np.all(ob[m[s]:] == SENTINEL)


def run_layer(w, max_tokens, seed=0, weight_in_down=False, fq=None):
    logits = synth.router_logits(w, seed, device="cuda")
    x = synth.hidden(w, seed, device="cuda")
    fp8 = w.dtype == "e4m3"
    w13, w2, s13, s2 = synth.expert_weights(w, seed, device="cuda")
    kw = {}
    if fp8:
        w13, w13s = moe.moe_quantize_weight_fp8(w13)
        w2, w2s = moe.moe_quantize_weight_fp8(w2)
        kw = dict(w13_scales=w13s, w2_scales=w2s)
        if s13 is not None:
            s13, s13s = moe.moe_quantize_weight_fp8(s13)
            s2, s2s = moe.moe_quantize_weight_fp8(s2)
            kw.update(shared_w13_scales=s13s, shared_w2_scales=s2s)
    layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, moe.MOE_E4M3 if fp8 else moe.MOE_BF16, w13=w13, w2=w2,
                         shared_w13=s13, shared_w2=s2, weight_in_down=weight_in_down, max_tokens=max_tokens, **kw)
    idx = torch.empty(w.T, w.K, dtype=torch.int32, device="cuda")
    wt = torch.empty(w.T, w.K, dtype=torch.float32, device="cuda")
    out = torch.full((w.T, w.H), SENTINEL, dtype=torch.int16).view(torch.bfloat16).cuda()
    n = torch.tensor([w.T_valid], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fqt = None if fq is None else torch.tensor([fq], dtype=torch.float32, device="cuda")
    layer.forward(x, out, idx, wt, logits=logits, num_tokens=n, dev_status=st, fq_scale=fqt)
    torch.cuda.synchronize()
    return out, st.item(), (logits, x, w13, w2, s13, s2, kw, idx, wt)


@pytest.mark.parametrize("case", ["tiny", "decode_small", "prefill_small_wd", "decode_fp8", "decode_full"])
def test_layer_batched_equals_contiguous(case):
    need_gpu()
    wd, fq = False, None
    if case == "tiny":
        w = WORKLOADS["tiny"]
        mt = w.T
    elif case == "decode_small":
        w = scaled(WORKLOADS["decode"], T=64, T_valid=64, H=512, I=256, E=32, K=4, dtype="bf16")
        mt = 72          # the shared block holds one row per token: 72 >= 64
    elif case == "prefill_small_wd":
        w = scaled(WORKLOADS["prefill"], T=128, T_valid=100, H=512, I=256, E=16, K=4)
        mt, wd, fq = 128, True, 30.0
    elif case == "decode_fp8":
        w = scaled(WORKLOADS["decode"], T=128, T_valid=128, H=1024, I=512, E=64, K=8)
        mt = 128
    else:
        w = WORKLOADS["decode"]          # full size: 257 blocks of 128 rows
        mt = w.T
    out_b, st_b, _ = run_layer(w, mt, weight_in_down=wd, fq=fq)
    out_c, st_c, _ = run_layer(w, 0, weight_in_down=wd, fq=fq)
    assert st_b == 0 and st_c == 0
    assert np.array_equal(bits(out_b), bits(out_c))


def test_layer_batched_matches_oracle():
    need_gpu()
    w = scaled(WORKLOADS["decode"], T=64, T_valid=64, H=512, I=256, E=32, K=4, dtype="bf16")
    out, st, (logits, x, w13, w2, s13, s2, _, idx, wt) = run_layer(w, 64)   # 64 tokens: the shared block needs 64 rows
    assert st == 0
    o_idx, o_w = ref.route_topk(host(logits), w.K, num_tokens=w.T_valid)
    assert np.array_equal(host(idx), o_idx)
    want = ref.layer_reference(bits(x), o_idx, o_w, ExpertBits(w13), ExpertBits(w2),
                               shared=(bits(s13), bits(s2)) if s13 is not None else None)
    got = bf16_bits_to_f32(bits(out)).astype(np.float64)
    assert ref.max_rel_err(got, want) <= 2e-2


def test_layer_batched_overflow_is_flagged():
    need_gpu()
    # 8 blocks of 6 rows for 64 tokens x top-2: most experts overflow
    w = scaled(WORKLOADS["tiny"], T=64, T_valid=64)
    out, st, _ = run_layer(w, 6)
    assert st & moe.MOE_DEV_OVERFLOW
    assert not np.any(bits(out) == SENTINEL)      # every token row is still written
