"""End-to-end GPU parity of moe_layer_forward against the oracle's dense per-token fp64
reference, on every workload at its full size (every one of the 8192 prefill tokens, every
decode token against both FP8 references) and on reduced sizes checked token by token; the FP8
workload against both the unquantised BF16 masters and the FP8-quantised operands; the
fake-quant workload with its calibration, captured and replayed in a CUDA graph after a
padding-only warm-up, with the on-device combine check.  Each comparison prints its max
relative error and its elementwise allclose fraction at atol = rtol = tolerance."""
import os

import numpy as np
import pytest
import torch

import combine_moe_route_softmax_gb300 as moe
from combine_moe_route_softmax_gb300 import synth
from combine_moe_route_softmax_gb300.synth import WORKLOADS, scaled
from gpu_helpers import ExpertBits, bits, host, need_gpu, sample_tokens
from oracle import moe_ref as ref
from oracle.formats import bf16_bits_to_f32

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "e4m3": 6e-2}
WORKERS = min(16, os.cpu_count() or 1)   # experts the oracle computes at once (threads)


class Setup:
    """A workload's inputs and weights on the GPU plus a MoeLayer over them."""

    def __init__(self, w, seed=0, weights=None, weight_tiles=False):
        self.w = w
        self.logits = synth.router_logits(w, seed, device="cuda")
        self.x = synth.hidden(w, seed, device="cuda")
        self.w13, self.w2, self.s13, self.s2 = weights or synth.expert_weights(w, seed, device="cuda")
        kw = {}
        if w.dtype == "e4m3":
            q13, sc13 = moe.moe_quantize_weight_fp8(self.w13)
            q2, sc2 = moe.moe_quantize_weight_fp8(self.w2)
            kw = dict(w13=q13, w2=q2, w13_scales=sc13, w2_scales=sc2)
            if w.shared:
                qs13, ss13 = moe.moe_quantize_weight_fp8(self.s13)
                qs2, ss2 = moe.moe_quantize_weight_fp8(self.s2)
                kw.update(shared_w13=qs13, shared_w2=qs2, shared_w13_scales=ss13, shared_w2_scales=ss2)
        else:
            kw = dict(w13=self.w13, w2=self.w2, shared_w13=self.s13, shared_w2=self.s2)
        self.layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, moe.MOE_E4M3 if w.dtype == "e4m3" else moe.MOE_BF16,
                                  weight_tiles=weight_tiles, **kw)
        self.topk_idx = torch.empty(w.T, w.K, dtype=torch.int32, device="cuda")
        self.topk_w = torch.empty(w.T, w.K, dtype=torch.float32, device="cuda")
        self.out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
        self.num_tokens = torch.tensor([w.T_valid], dtype=torch.int32, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        # oracle routing (+ the workload's slot padding) from the same logits
        self.o_idx, self.o_w = ref.route_topk(host(self.logits), w.K, num_tokens=w.T_valid)
        if w.slot_pad > 0:
            pad = host(synth.slot_padding(w, seed, device="cuda"))
            self.o_idx = np.where(pad, -1, self.o_idx).astype(np.int32)
            self.o_w = np.where(pad, 0, self.o_w).astype(np.float32)

    def forward(self, fq_scale=None):
        if self.w.slot_pad > 0:     # routed outside the layer, padding slots set by the caller
            self.topk_idx.copy_(torch.from_numpy(self.o_idx))
            self.topk_w.copy_(torch.from_numpy(self.o_w))
            return self.layer.forward(self.x, self.out, self.topk_idx, self.topk_w, fq_scale=fq_scale,
                                      dev_status=self.status)
        return self.layer.forward(self.x, self.out, self.topk_idx, self.topk_w, logits=self.logits,
                                  num_tokens=self.num_tokens, fq_scale=fq_scale, dev_status=self.status)

    def reference(self, tokens, fp8=None, fq_scale=None):
        shared = (bits(self.s13), bits(self.s2)) if self.w.shared else None
        return ref.layer_reference(bits(self.x), self.o_idx, self.o_w, ExpertBits(self.w13), ExpertBits(self.w2),
                                   shared=shared, tokens=tokens, fq_scale=fq_scale,
                                   fp8=(self.w.dtype == "e4m3") if fp8 is None else fp8, workers=WORKERS)


def allclose_fraction(got, want, tol):
    """Share of elements with |got - want| <= tol + tol * |want| (the elementwise allclose
    at atol = rtol = tol of the MoonEP page's test)."""
    return float(np.mean(np.abs(got - want) <= tol + tol * np.abs(want)))


def report(label, got, want, tol):
    """Both error figures of one comparison, printed on one line (pytest -s or -rP shows
    them); returns (max relative error, allclose fraction)."""
    err = ref.max_rel_err(got, want)
    frac = allclose_fraction(got, want, tol)
    print(f"{label}: max rel err {err:.4e}, allclose(atol=rtol={tol:g}) fraction {frac:.6f} "
          f"over {got.shape[0]} tokens x {got.shape[1]} columns")
    return err, frac


def check_layer(s, tokens, tol, fq_scale_dev=None, fq_scale_ref=None, label=None):
    s.forward(fq_scale_dev)
    torch.cuda.synchronize()
    assert s.status.item() == 0
    if s.w.slot_pad == 0:
        assert np.array_equal(host(s.topk_idx), s.o_idx)
    got = bf16_bits_to_f32(bits(s.out)).astype(np.float64)
    want = s.reference(tokens, fq_scale=fq_scale_ref)
    err, _ = report(label or s.w.name, got[tokens], want, tol)
    assert err <= tol, err
    # padding rows of the bucket are +0
    assert np.all(bits(s.out)[s.w.T_valid:] == 0)
    return err


@pytest.mark.parametrize("name,T,H,I,E,K", [
    ("tiny", None, None, None, None, None),
    ("mid", None, None, None, None, None),
    ("prefill", 96, 512, 256, 16, 4),          # the prefill shape family, reduced: every token checked
    ("decode", 64, 1024, 512, 16, 4),          # FP8 with a shared expert, reduced: every token checked
])
def test_layer_every_token(name, T, H, I, E, K):
    need_gpu()
    w = WORKLOADS[name]
    if T is not None:
        w = scaled(w, T=T, T_valid=T * 3 // 4 if name == "prefill" else T, H=H, I=I, E=E, K=K)
    s = Setup(w)
    tokens = np.arange(w.T_valid)
    check_layer(s, tokens, TOL[w.dtype])


def test_layer_prefill_full_size_every_token():
    """Full prefill size, in the benchmark's configuration (weights in the tile layout): all
    8192 tokens against the fp64 reference (the whole layer output is also checked as the
    re-sum of the layer's own expert rows)."""
    need_gpu()
    s = Setup(WORKLOADS["prefill"], weight_tiles=True)
    check_layer(s, np.arange(8192), TOL["bf16"], label="prefill (every token)")
    # the expert-major layout the layer built is the oracle's, bit for bit
    v = s.layer.views
    cap = 16384 * 8 + 16384
    cu, src, inv, smap, _ = ref.permute(s.o_idx, 256, with_shared=True)
    assert np.array_equal(host(s.layer.view("cu_seqlens", (258,), torch.int32)), cu)
    assert np.array_equal(host(s.layer.view("src_row", (cap,), torch.int32)), src)
    assert np.array_equal(host(s.layer.view("inv_map", (16384, 8), torch.int32)), inv)
    assert v.cap == cap
    # every token: the output is the fixed-order re-sum of the layer's own expert rows
    H = 7168
    y = s.layer.view("y", (cap, H), torch.bfloat16)
    vs = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_combine_verify(y, s.layer.view("inv_map", (16384, 8), torch.int32), s.topk_w, s.out, vs, shared_y=y,
                           shared_map=s.layer.view("shared_map", (16384,), torch.int32))
    torch.cuda.synchronize()
    assert vs.item() == 0
    # expert rows of 48 distinct experts (and the shared expert), each against the oracle's
    # SwiGLU expert on its token: every grouped-GEMM segment kind, checked row by row
    rng = np.random.default_rng(3)
    n_routed = int(cu[256])
    seg_of = np.searchsorted(cu, np.arange(int(cu[-1])), side="right") - 1
    experts = rng.choice(np.unique(seg_of[:n_routed]), size=48, replace=False)
    rows = [int(rng.choice(np.nonzero(seg_of == e)[0])) for e in experts]
    rows.append(int(rng.integers(n_routed, int(cu[-1]))))              # a shared-expert row
    xb = bits(s.x)
    yb = bits(y)
    for r in rows:
        e = int(seg_of[r])
        tok = int(ref.row_tokens(src[r:r + 1], 16384, 8)[0])
        f = lambda t: bf16_bits_to_f32(t).astype(np.float64)
        w13, w2 = (bits(s.s13), bits(s.s2)) if e == 256 else (bits(s.w13[e]), bits(s.w2[e]))
        want = ref.swiglu_expert(f(xb[tok:tok + 1]), f(w13), f(w2))[0]
        got = bf16_bits_to_f32(yb[r]).astype(np.float64)
        assert ref.max_rel_err(got, want) <= TOL["bf16"], (r, e)


def test_layer_decode_full_size_every_token():
    """Full decode size, every one of the 128 tokens compared twice: against the fp64 layer
    on the FP8-quantised operands at the FP8 tolerance 6e-2 (every touched expert's weights
    quantised by the oracle), and against the fp64 layer on the unquantised BF16 masters at
    the bound E4M3's rounding allows (below).  The 6e-2 figure is the MoonEP page's test
    tolerance ("BF16 integration of MoonEP balanced EP backend", Test Result: atol = rtol =
    6e-2 against a per-token reference MoE), set there for BF16 operands.  Weights in the
    tile layout, as the benchmark runs."""
    need_gpu()
    s = Setup(WORKLOADS["decode"], weight_tiles=True)
    check_layer(s, np.arange(128), TOL["e4m3"], label="decode vs the FP8-operand reference")
    # Against the BF16 masters the difference is E4M3's own rounding: x, W13, h and W2 are
    # each rounded with a relative error of rms 2^-4 / sqrt(3) = 3.6 % (three mantissa
    # bits), which compounds to sqrt(4) * 3.6 % = 7.2 % rms on the output.  The oracle's FP8
    # reference itself sits 6.4 % rms / 6.9 % max-relative from the masters on these shapes,
    # so the 6e-2 bound cannot hold here by construction; the gate is that derived rms
    # bound (with a margin to 8 %) and a max-relative bound of 0.10, both printed.
    tokens = np.arange(128)
    got = bf16_bits_to_f32(bits(s.out)).astype(np.float64)
    want = s.reference(tokens, fp8=False)
    err_master, _ = report("decode vs the BF16-master reference", got, want, TOL["e4m3"])
    rms = float(np.sqrt(((got - want) ** 2).mean() / (want ** 2).mean()))
    print(f"decode vs the BF16-master reference: rms relative error {rms:.4e}")
    assert rms <= 8e-2, rms
    assert err_master <= 0.10, err_master
    # every token: the output is the fixed-order re-sum of the layer's own expert rows, and
    # the layout is the oracle's
    cap = 128 * 8 + 128
    y = s.layer.view("y", (cap, 7168), torch.bfloat16)
    inv = s.layer.view("inv_map", (128, 8), torch.int32)
    smap = s.layer.view("shared_map", (128,), torch.int32)
    vs = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_combine_verify(y, inv, s.topk_w, s.out, vs, shared_y=y, shared_map=smap)
    torch.cuda.synchronize()
    assert vs.item() == 0
    cu, src, o_inv, o_smap, _ = ref.permute(s.o_idx, 256, with_shared=True)
    assert np.array_equal(host(inv), o_inv) and np.array_equal(host(smap), o_smap)


def calibrate(w, seed, weights):
    """Calibration batch (16 tokens drawn with seed + 1, the layer's own weights): GPU amax
    over the layer's weighted routed rows, and the oracle's amax over its own rows."""
    wc = scaled(w, T=16, T_valid=16, fake_quant=False, graph=False)
    c = Setup(wc, seed=seed + 1, weights=weights)
    c.forward()
    T, K, cap = wc.T, wc.K, c.layer.views.cap
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    moe.moe_combine_amax(c.layer.view("y", (cap, w.H), torch.bfloat16), c.layer.view("inv_map", (T, K), torch.int32),
                         c.topk_w, amax)
    s_gpu = moe.moe_fq_scale_from_amax(amax)
    # oracle: every valid weighted row r = w_k * expert(x_t), as float32
    best = np.float32(0)
    x = bf16_bits_to_f32(bits(c.x)).astype(np.float64)
    for e in np.unique(c.o_idx[c.o_idx >= 0]):
        where = np.nonzero(c.o_idx == e)
        ye = ref.swiglu_expert(x[where[0]], bf16_bits_to_f32(bits(c.w13[int(e)])), bf16_bits_to_f32(bits(c.w2[int(e)])))
        r = (c.o_w[where][:, None].astype(np.float64) * ye).astype(np.float32)
        best = max(best, np.float32(np.abs(r).max()))
    s_o = ref.fq_scale_from_amax(best)
    return s_gpu, float(s_o), float(host(amax)[0]), float(best)


def test_fake_quant_layer_in_cuda_graph():
    need_gpu()
    w = WORKLOADS["prefill_fq"]
    weights = synth.expert_weights(w, 0, device="cuda")
    s_gpu, s_o, a_gpu, a_o = calibrate(w, 0, weights)
    assert abs(a_gpu - a_o) <= 1e-2 * a_o, (a_gpu, a_o)
    s = Setup(w, weights=weights)
    # warm-up with a padding-only batch (all rows past num_tokens = 0 are padding)
    s.num_tokens.fill_(0)
    s.forward(s_gpu)
    torch.cuda.synchronize()
    assert np.all(bits(s.out) == 0)
    verify_status = torch.zeros(1, dtype=torch.int32, device="cuda")
    T, K, H, cap = w.T, w.K, w.H, s.layer.views.cap
    y = s.layer.view("y", (cap, H), torch.bfloat16)
    inv = s.layer.view("inv_map", (T, K), torch.int32)
    smap = s.layer.view("shared_map", (T,), torch.int32)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        s.forward(s_gpu)
        moe.moe_combine_verify(y, inv, s.topk_w, s.out, verify_status, shared_y=y, shared_map=smap, fq_scale=s_gpu)
    s.num_tokens.fill_(w.T_valid)
    g.replay()
    torch.cuda.synchronize()
    assert verify_status.item() == 0 and s.status.item() == 0
    graph_out = bits(s.out).copy()
    # eager run of the same batch is bit-identical to the replay
    s.forward(s_gpu)
    torch.cuda.synchronize()
    assert np.array_equal(bits(s.out), graph_out)
    assert np.array_equal(host(s.topk_idx), s.o_idx)
    tokens = np.arange(8192)
    got = bf16_bits_to_f32(graph_out).astype(np.float64)[tokens]
    want = s.reference(tokens, fq_scale=np.float32(s_o))
    err, _ = report("prefill_fq graph replay (every token)", got, want, TOL["e4m3"])
    assert err <= TOL["e4m3"], err
    # fake-quant changed the output (on a sample of tokens)
    few = sample_tokens(8192, 64, seed=3)
    assert ref.max_rel_err(want[few], s.reference(few)) > 1e-3
    # a graph holding only the on-device check: rows that no longer reproduce the output
    # (a changed layout) set the mismatch bit on replay instead of asserting
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        moe.moe_combine_verify(y, inv, s.topk_w, s.out, verify_status, shared_y=y, shared_map=smap, fq_scale=s_gpu)
    g2.replay()
    torch.cuda.synchronize()
    assert verify_status.item() == 0
    y.view(torch.int16)[int(host(inv)[0, 0]), 0] ^= 0x40
    g2.replay()
    torch.cuda.synchronize()
    assert verify_status.item() == moe.MOE_DEV_VERIFY_MISMATCH
