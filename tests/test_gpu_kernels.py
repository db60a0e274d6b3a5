"""GPU parity of the index and data-movement steps against the CPU oracle, through the C
ABI: route (ids bit-exact, weights within a few float32 ulp), permute (every index array
and every gathered row bit-exact, BF16 and E4M3), FP8 quantisers (bit-exact) and the
fixed-order combine (bit-exact, with and without shared rows and fake-quant), at small
ragged sizes, edge cases and the workloads' full sizes."""
import numpy as np
import pytest
import torch

import combine_moe_route_softmax_gb300 as moe
from combine_moe_route_softmax_gb300 import synth
from combine_moe_route_softmax_gb300.synth import WORKLOADS
from golden_cases import build, load_cases
from gpu_helpers import bits, host, need_gpu
from oracle import moe_ref as ref
from oracle.formats import bf16_bits_to_f32

pytestmark = pytest.mark.gpu

FULL = ["tiny", "mid", "decode", "prefill"]


def dev_status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def routed(w, seed=0, device="cuda"):
    """Oracle routing of the workload's logits (+ its slot padding), as numpy."""
    logits = synth.router_logits(w, seed, device=device)
    idx, wt = ref.route_topk(host(logits), w.K, num_tokens=w.T_valid)
    if w.slot_pad > 0:
        pad = host(synth.slot_padding(w, seed, device=device))
        idx = np.where(pad, -1, idx).astype(np.int32)
        wt = np.where(pad, 0, wt).astype(np.float32)
    return logits, idx, wt


# ----------------------------------------------------------------------------- route
@pytest.mark.parametrize("name", FULL)
def test_route_matches_oracle(name):
    need_gpu()
    w = WORKLOADS[name]
    logits = synth.router_logits(w, 0, device="cuda")
    n = torch.tensor([w.T_valid], dtype=torch.int32, device="cuda")
    idx, wt = moe.moe_route_topk(logits, w.K, num_tokens=n)
    oi, ow = ref.route_topk(host(logits), w.K, num_tokens=w.T_valid)
    assert np.array_equal(host(idx), oi)
    gw = host(wt).astype(np.float64)
    assert np.all(gw[w.T_valid:] == 0)
    rel = np.abs(gw - ow) / np.maximum(np.abs(ow), 1e-30)
    assert rel[: w.T_valid].max() <= 4 * 2.0 ** -24 * w.K   # a few float32 ulp (expf, sum, divide)


def test_route_ties_and_small_shapes():
    need_gpu()
    logits = torch.zeros(5, 40, device="cuda")
    logits[1, [7, 33, 39]] = 2.0
    logits[2] = torch.arange(40, device="cuda", dtype=torch.float32).flip(0)
    idx, wt = moe.moe_route_topk(logits, 4)
    oi, ow = ref.route_topk(host(logits), 4)
    assert np.array_equal(host(idx), oi)
    assert host(idx)[0].tolist() == [0, 1, 2, 3] and host(idx)[1].tolist() == [7, 33, 39, 0]
    assert np.allclose(host(wt), ow, rtol=1e-6)
    # signed zeros are equal logits: the lower id comes first
    z = torch.zeros(2, 40, device="cuda")
    z[0, [3, 9, 20]] = -0.0
    z[0, [5, 11]] = 1.0
    z[1, :] = -0.0
    z[1, 17] = 0.0
    idx, _ = moe.moe_route_topk(z, 4)
    oi, _ = ref.route_topk(host(z), 4)
    assert np.array_equal(host(idx), oi) and host(idx)[0].tolist() == [5, 11, 0, 1]
    assert host(idx)[1].tolist() == [0, 1, 2, 3]
    for E, K in [(1, 1), (32, 32), (33, 5), (300, 6), (1024, 8), (700, 32)]:
        lg = torch.randn(17, E, device="cuda", generator=torch.Generator("cuda").manual_seed(E))
        idx, wt = moe.moe_route_topk(lg, K)
        oi, ow = ref.route_topk(host(lg), K)
        assert np.array_equal(host(idx), oi)
        assert np.allclose(host(wt), ow, rtol=1e-6)


# --------------------------------------------------------------------------- permute
def check_permute(idx_np, E, x, with_shared, out_dtype=moe.MOE_BF16, expect_status=0):
    T, K = idx_np.shape
    st = dev_status()
    res = moe.moe_permute(torch.from_numpy(idx_np).cuda(), E, x, with_shared=with_shared, out_dtype=out_dtype,
                          dev_status=st)
    cu, src, inv, smap, ost = ref.permute(idx_np, E, with_shared=with_shared)
    torch.cuda.synchronize()
    assert int(st.item()) == ost == expect_status
    assert np.array_equal(host(res["cu_seqlens"]), cu)
    assert np.array_equal(host(res["src_row"]), src)
    assert np.array_equal(host(res["inv_map"]), inv)
    if with_shared:
        assert np.array_equal(host(res["shared_map"]), smap)
    N = int(cu[-1])
    xb = bits(x)
    want = ref.gather_rows(xb, src[:N], T, K) if N else np.zeros((0, x.shape[1]), np.uint16)
    if out_dtype == moe.MOE_BF16:
        assert np.array_equal(bits(res["xp"][:N]), want)
    else:
        q, s = ref.act_quant_1x128(bf16_bits_to_f32(want))
        assert np.array_equal(host(res["xp"][:N]), q)
        assert np.array_equal(host(res["xp_scales"][:N]), s)
    return res, N


@pytest.mark.parametrize("name,with_shared,dt", [("tiny", False, moe.MOE_BF16), ("mid", False, moe.MOE_BF16),
                                                 ("mid", True, moe.MOE_BF16), ("decode", True, moe.MOE_E4M3),
                                                 ("prefill", True, moe.MOE_BF16)])
def test_permute_matches_oracle(name, with_shared, dt):
    need_gpu()
    w = WORKLOADS[name]
    _, idx, _ = routed(w)
    x = synth.hidden(w, 0, device="cuda")
    check_permute(idx, w.E, x, with_shared, dt)


@pytest.mark.parametrize("T,K,E,pad,shared", [(1, 1, 1, 0.0, True), (1000, 3, 5, 0.3, True), (65, 8, 256, 0.1, False),
                                              (130, 6, 1024, 0.0, True), (7, 2, 2, 0.9, True)])
def test_permute_ragged_and_edge_shapes(T, K, E, pad, shared):
    need_gpu()
    rng = np.random.default_rng(T * 7 + K)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[rng.random((T, K)) < pad] = -1
    x = torch.randn(T, 384, generator=torch.Generator().manual_seed(T)).to(torch.bfloat16).cuda()
    check_permute(idx, E, x, shared, moe.MOE_BF16)
    check_permute(idx, E, x, shared, moe.MOE_E4M3)


@pytest.mark.parametrize("T,H", [(1, 7168), (3, 7168), (130, 7168), (9, 1152), (200, 2048)])
def test_permute_few_tokens_split_columns(T, H):
    """Few tokens: each token's columns are gathered by several warps (parts of whole
    vector groups; H = 1152 leaves a partial last group)."""
    need_gpu()
    rng = np.random.default_rng(T + H)
    E, K = 40, 6
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[rng.random((T, K)) < 0.1] = -1
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(H)).to(torch.bfloat16).cuda()
    check_permute(idx, E, x, True, moe.MOE_BF16)
    check_permute(idx, E, x, True, moe.MOE_E4M3)


def test_permute_all_padding_and_bad_ids():
    need_gpu()
    x = torch.randn(64, 256).to(torch.bfloat16).cuda()
    res, N = check_permute(np.full((64, 4), -1, np.int32), 16, x, True)
    assert N == 0
    idx = np.array([[0, 5], [-2, 1], [1, -1], [3, 4]], np.int32)
    check_permute(idx, 4, x[:4], True, expect_status=moe.MOE_DEV_BAD_EXPERT)


def test_permute_workspace_too_small_is_rejected():
    need_gpu()
    x = torch.randn(64, 256).to(torch.bfloat16).cuda()
    idx = torch.zeros(64, 2, dtype=torch.int32, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_permute(idx, 8, x, ws=small)
    assert e.value.code == 2


# ---------------------------------------------------------------------------- quant
def test_quantize_act_and_weight_bit_exact():
    need_gpu()
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(300, 1024, generator=g) * torch.exp2(torch.randint(-8, 8, (300, 1), generator=g))).to(torch.bfloat16)
    x[7, 256:384] = 0
    q, s = moe.moe_quantize_act_fp8(x.cuda())
    oq, os_ = ref.act_quant_1x128(bf16_bits_to_f32(bits(x)))
    assert np.array_equal(host(q), oq) and np.array_equal(host(s), os_)
    wt = (torch.randn(3, 256, 384, generator=g) * 0.03).to(torch.bfloat16)
    wt[1, 128:, :128] = 0
    q, s = moe.moe_quantize_weight_fp8(wt.cuda())
    for m in range(3):
        oq, os_ = ref.weight_quant_128x128(bf16_bits_to_f32(bits(wt[m])))
        assert np.array_equal(host(q[m]), oq) and np.array_equal(host(s[m]), os_)


# --------------------------------------------------------------------------- combine
@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c["name"])
def test_combine_golden_cases_on_gpu(case):
    need_gpu()
    c = build(case)
    y = torch.from_numpy(c["y"].view(np.int16)).cuda().view(torch.bfloat16)
    inv = torch.from_numpy(c["inv_map"]).cuda()
    w = torch.from_numpy(c["w"]).cuda()
    shared = None if c["shared"] is None else torch.from_numpy(c["shared"].view(np.int16)).cuda().view(torch.bfloat16)
    fq = None if c["fq_scale"] is None else torch.tensor([c["fq_scale"]], dtype=torch.float32, device="cuda")
    out = moe.moe_combine(y, inv, w, shared_y=shared, fq_scale=fq)
    assert np.all(bits(out) == c["expect"])


def combine_problem(T, K, E, H, pad, shared, seed, device="cuda"):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[rng.random((T, K)) < pad] = -1
    cu, src, inv, smap, _ = ref.permute(idx, E, with_shared=shared)
    cap = len(src)
    g = torch.Generator(device).manual_seed(seed)
    y = torch.randn(cap, H, generator=g, device=device).to(torch.bfloat16)
    wt = torch.rand(T, K, generator=g, device=device)
    return idx, inv, smap, y, wt


@pytest.mark.parametrize("T,K,E,H,pad,shared,fq", [(333, 8, 64, 1024, 0.1, True, None), (333, 8, 64, 1024, 0.1, True, 37.5),
                                                   (50, 2, 8, 256, 0.0, False, None), (64, 12, 16, 384, 0.2, True, 3.0),
                                                   (16384, 8, 256, 7168, 0.0, True, None),
                                                   # few tokens: each row split over several warps (uneven parts)
                                                   (1, 8, 64, 7168, 0.0, True, 12.0), (5, 8, 64, 7168, 0.1, True, None),
                                                   (130, 8, 256, 7168, 0.0, True, None), (7, 4, 9, 1152, 0.2, False, 3.0)])
def test_combine_bit_exact(T, K, E, H, pad, shared, fq):
    need_gpu()
    idx, inv, smap, y, wt = combine_problem(T, K, E, H, pad, shared, seed=T + K)
    if T == 16384:       # the prefill bucket: rows past 8192 are padding tokens
        inv[8192:] = -1
        if smap is not None:
            smap[8192:] = -1
    fqt = None if fq is None else torch.tensor([fq], dtype=torch.float32, device="cuda")
    out = moe.moe_combine(y, torch.from_numpy(inv).cuda(), wt, shared_y=y if shared else None,
                          shared_map=torch.from_numpy(smap).cuda() if shared else None, fq_scale=fqt)
    yb = bits(y)
    want = ref.combine(yb, inv, host(wt), shared_bits=yb if shared else None, shared_map=smap, fq_scale=fq)
    assert np.array_equal(bits(out), want)


def test_combine_dense_shared_rows_and_verify():
    need_gpu()
    T, K, E, H = 200, 4, 16, 512
    idx, inv, _, y, wt = combine_problem(T, K, E, H, 0.25, False, seed=3)
    inv[5] = -1
    ys = torch.randn(T, H, generator=torch.Generator("cuda").manual_seed(9), device="cuda").to(torch.bfloat16)
    invd = torch.from_numpy(inv).cuda()
    out = moe.moe_combine(y, invd, wt, shared_y=ys)
    want = ref.combine(bits(y), inv, host(wt), shared_bits=bits(ys))
    assert np.array_equal(bits(out), want)
    assert np.all(bits(out)[5] == 0)
    st = dev_status()
    moe.moe_combine_verify(y, invd, wt, out, st, shared_y=ys)
    torch.cuda.synchronize()
    assert st.item() == 0
    bad = out.clone()
    bad.view(torch.int16)[17, 3] ^= 1
    moe.moe_combine_verify(y, invd, wt, bad, st, shared_y=ys)
    torch.cuda.synchronize()
    assert st.item() == moe.MOE_DEV_VERIFY_MISMATCH


def test_combine_amax_and_scale():
    need_gpu()
    T, K, E, H = 300, 8, 32, 1024
    idx, inv, _, y, wt = combine_problem(T, K, E, H, 0.1, False, seed=4)
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    moe.moe_combine_amax(y, torch.from_numpy(inv).cuda(), wt, amax)
    s = moe.moe_fq_scale_from_amax(amax)
    oa = ref.combine_amax(bits(y), inv, host(wt))
    assert host(amax)[0] == oa
    assert host(s)[0] == ref.fq_scale_from_amax(oa)
