"""GPU parity of the layer's options against the oracle: dispatch fake-quant (routed rows
fake-quantised with a calibrated per-tensor E4M3 scale, shared rows untouched), router
weights applied in the down projection (rows stored weighted, the combine only sums), and
their building blocks (moe_permute_ex, moe_grouped_gemm_ex row scale, combine without
weights, moe_amax_bf16)."""
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


def random_idx(T, K, E, pad, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[rng.random((T, K)) < pad] = -1
    return idx


def test_amax_bf16_and_scale_bit_exact():
    need_gpu()
    x = (torch.randn(1000, 1024, generator=torch.Generator().manual_seed(1)) * 3).to(torch.bfloat16)
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    moe.moe_amax_bf16(x.cuda(), amax)
    s = moe.moe_fq_scale_from_amax(amax)
    oa = ref.tensor_amax(bits(x))
    assert host(amax)[0] == oa and host(s)[0] == ref.fq_scale_from_amax(oa)


@pytest.mark.parametrize("shared", [False, True])
def test_permute_ex_dispatch_fake_quant_and_row_weights(shared):
    need_gpu()
    T, K, E, H = 300, 6, 24, 512
    idx = random_idx(T, K, E, 0.15, seed=7)
    g = torch.Generator().manual_seed(8)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    topk_w = torch.rand(T, K, generator=g)
    s = np.float32(448.0) / ref.tensor_amax(bits(x))
    res = moe.moe_permute(torch.from_numpy(idx).cuda(), E, x.cuda(), with_shared=shared,
                          dispatch_scale=torch.tensor([s], device="cuda"), topk_w=topk_w.cuda())
    cu, src, inv, smap, _ = ref.permute(idx, E, with_shared=shared)
    assert np.array_equal(host(res["cu_seqlens"]), cu) and np.array_equal(host(res["src_row"]), src)
    n_routed, N = int(cu[E]), int(cu[-1])
    tok = ref.row_tokens(src[:N], T, K)
    xq = ref.dispatch_qdq_bits(bits(x), s)
    got = bits(res["xp"][:N])
    assert np.array_equal(got[:n_routed], xq[tok[:n_routed]])            # routed rows: fake-quantised
    assert np.array_equal(got[n_routed:], bits(x)[tok[n_routed:]])       # shared rows: original
    rw = host(res["row_weights"][:N])
    assert np.array_equal(rw[:n_routed], host(topk_w).reshape(-1)[src[:n_routed]])
    assert np.all(rw[n_routed:] == 1.0)


@pytest.mark.parametrize("fp8", [False, True])
def test_grouped_gemm_row_scale(fp8):
    need_gpu()
    cu = [0, 5, 300, 300, 517]
    rows, k, n, E = 560, 256, 384, 4
    g = torch.Generator().manual_seed(9)
    a = torch.randn(rows, k, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, n, k, generator=g) / k ** 0.5).to(torch.bfloat16)
    rs = torch.rand(rows, generator=g)
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    if fp8:
        qa, sa = ref.act_quant_1x128(bf16_bits_to_f32(bits(a)))
        qw, sw = zip(*[ref.weight_quant_128x128(bf16_bits_to_f32(bits(w[i]))) for i in range(E)])
        qw, sw = np.stack(qw), np.stack(sw)
        T_ = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()
        out, _ = moe.moe_grouped_gemm(T_(qa), cu_t, T_(qw), a_scales=T_(sa), w_scales=T_(sw), row_scale=rs.cuda())
        a64 = ref.dequant(qa, sa, 1)
        wl = [ref.dequant(qw[e], sw[e], 128) for e in range(E)]
    else:
        out, _ = moe.moe_grouped_gemm(a.cuda(), cu_t, w.cuda(), row_scale=rs.cuda())
        f = lambda t: bf16_bits_to_f32(bits(t)).astype(np.float64)
        a64, wl = f(a), [f(w[e]) for e in range(E)]
    want = np.concatenate([a64[cu[e]:cu[e + 1]] @ wl[e].T for e in range(E)]) * host(rs)[:cu[-1], None]
    got = bf16_bits_to_f32(bits(out))[:cu[-1]].astype(np.float64)
    scale = np.abs(want).max()
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 2e-3 * scale)


@pytest.mark.parametrize("fq", [None, 60.0])
def test_combine_of_preweighted_rows_bit_exact(fq):
    need_gpu()
    T, K, E, H = 333, 8, 64, 1024
    idx = random_idx(T, K, E, 0.1, seed=10)
    cu, src, inv, smap, _ = ref.permute(idx, E, with_shared=True)
    y = torch.randn(len(src), H, generator=torch.Generator().manual_seed(11)).to(torch.bfloat16)
    fqt = None if fq is None else torch.tensor([fq], dtype=torch.float32, device="cuda")
    yc = y.cuda()
    out = moe.moe_combine(yc, torch.from_numpy(inv).cuda(), None, shared_y=yc,
                          shared_map=torch.from_numpy(smap).cuda(), fq_scale=fqt)
    want = ref.combine(bits(y), inv, None, shared_bits=bits(y), shared_map=smap, fq_scale=fq)
    assert np.array_equal(bits(out), want)


def layer_case(w, weight_in_down=False, dispatch=False, seed=0):
    logits = synth.router_logits(w, seed, device="cuda")
    x = synth.hidden(w, seed, device="cuda")
    w13, w2, s13, s2 = synth.expert_weights(w, seed, device="cuda")
    layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, moe.MOE_BF16, w13=w13, w2=w2, shared_w13=s13, shared_w2=s2,
                         weight_in_down=weight_in_down)
    idx = torch.empty(w.T, w.K, dtype=torch.int32, device="cuda")
    wt = torch.empty(w.T, w.K, dtype=torch.float32, device="cuda")
    out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    n = torch.tensor([w.T_valid], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ds, o_s = None, None
    if dispatch:
        # calibration on the batch's own tokens (the real rows of the bucket)
        amax = torch.zeros(1, dtype=torch.float32, device="cuda")
        moe.moe_amax_bf16(x[:w.T_valid].contiguous(), amax)
        ds = moe.moe_fq_scale_from_amax(amax)
        o_s = ref.fq_scale_from_amax(ref.tensor_amax(bits(x[:w.T_valid])))
        assert host(ds)[0] == o_s
    layer.forward(x, out, idx, wt, logits=logits, num_tokens=n, dev_status=status, dispatch_scale=ds)
    torch.cuda.synchronize()
    assert status.item() == 0
    o_idx, o_w = ref.route_topk(host(logits), w.K, num_tokens=w.T_valid)
    assert np.array_equal(host(idx), o_idx)
    shared = (bits(s13), bits(s2)) if w.shared else None
    want = ref.layer_reference(bits(x), o_idx, o_w, ExpertBits(w13), ExpertBits(w2), shared=shared,
                               tokens=np.arange(w.T_valid), dispatch_scale=o_s)
    got = bf16_bits_to_f32(bits(out)).astype(np.float64)
    return ref.max_rel_err(got[:w.T_valid], want), got, out, layer


@pytest.mark.parametrize("name", ["tiny", "prefill"])
def test_layer_router_weight_in_down_projection(name):
    need_gpu()
    w = WORKLOADS[name]
    if name == "prefill":
        w = scaled(w, T=96, T_valid=72, H=512, I=256, E=16, K=4)
    err, got, out, layer = layer_case(w, weight_in_down=True)
    assert err <= 2e-2, err
    assert np.all(bits(out)[w.T_valid:] == 0)
    # the combine of the stored (weighted) rows reproduces the output bit for bit
    v, d = layer.views, layer.desc
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = layer.view("y", (v.cap, d.H), torch.bfloat16)
    inv = layer.view("inv_map", (d.T, d.K), torch.int32)
    smap = layer.view("shared_map", (d.T,), torch.int32) if d.has_shared else None
    moe.moe_combine_verify(y, inv, None, out, st, shared_y=y if d.has_shared else None, shared_map=smap)
    torch.cuda.synchronize()
    assert st.item() == 0


def test_layer_dispatch_fake_quant():
    need_gpu()
    w = scaled(WORKLOADS["prefill"], T=96, T_valid=72, H=512, I=256, E=16, K=4)
    err, got, _, _ = layer_case(w, dispatch=True)
    assert err <= 2e-2, err
    # the option changes the output: the plain layer differs from the fake-quantised one
    err_plain, got_plain, _, _ = layer_case(w)
    assert err_plain <= 2e-2
    assert ref.max_rel_err(got, got_plain) > 1e-3


def test_dispatch_fake_quant_rejected_for_e4m3_layers():
    need_gpu()
    x = torch.zeros(16, 256, dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(16, 2, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_permute(idx, 4, x, out_dtype=moe.MOE_E4M3, dispatch_scale=torch.ones(1, device="cuda"))
    assert e.value.code == 3


@pytest.mark.parametrize("full", [False, True], ids=["reduced", "full"])
@pytest.mark.parametrize("weight_in_down", [False, True])
def test_layer_gemm_pairs_bit_identical(weight_in_down, full):
    """gemm_pairs runs both grouped GEMMs on SM pairs: the layer output equals the default
    layer's bit for bit (prefill shapes, reduced and full size, with the shared expert and the
    skewed routing that gives long and short segments; at full size both computations run
    streaming CTAs); E4M3, the batched layout and the fused combine are refused."""
    need_gpu()
    if full and weight_in_down:
        pytest.skip("one full-size case is enough")
    w = WORKLOADS["prefill"] if full else scaled(WORKLOADS["prefill"], T=1024, T_valid=768, E=32)
    logits = synth.router_logits(w, 0, device="cuda")
    x = synth.hidden(w, 0, device="cuda")
    w13, w2, s13, s2 = synth.expert_weights(w, 0, device="cuda")
    outs = []
    for pairs in (False, True):
        layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, moe.MOE_BF16, w13=w13, w2=w2, shared_w13=s13, shared_w2=s2,
                             weight_in_down=weight_in_down, gemm_pairs=pairs)
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
    for kw in (dict(max_tokens=w.T), dict(fuse_combine=True)):
        bad = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, moe.MOE_BF16, w13=w13, w2=w2, shared_w13=s13, shared_w2=s2,
                           gemm_pairs=True, **kw)
        with pytest.raises(moe.MoeError):
            bad.forward(x, outs[0], torch.empty(w.T, w.K, dtype=torch.int32, device="cuda"),
                        torch.empty(w.T, w.K, dtype=torch.float32, device="cuda"), logits=logits)
