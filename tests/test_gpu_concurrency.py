"""Concurrent use: two layers (BF16 and E4M3, different shapes) driven from two host threads
on two CUDA streams at once give, call after call, the bits each gives alone (the library's
host-side state -- per-device SM counts, kernel attributes, the tensor-map encoder -- is
shared and must tolerate it; ctypes releases the GIL around every call)."""
import threading

import numpy as np
import pytest
import torch

import combine_moe_route_softmax_gb300 as moe
from combine_moe_route_softmax_gb300 import synth
from combine_moe_route_softmax_gb300.synth import WORKLOADS, scaled
from gpu_helpers import bits, need_gpu

pytestmark = pytest.mark.gpu


def make(w, fp8):
    x = synth.hidden(w, 0, device="cuda")
    logits = synth.router_logits(w, 0, device="cuda")
    w13, w2, s13, s2 = synth.expert_weights(w, 0, device="cuda")
    kw = dict(w13=w13, w2=w2, shared_w13=s13, shared_w2=s2)
    if fp8:
        q13, c13 = moe.moe_quantize_weight_fp8(w13)
        q2, c2 = moe.moe_quantize_weight_fp8(w2)
        a, b = moe.moe_quantize_weight_fp8(s13)
        c, d = moe.moe_quantize_weight_fp8(s2)
        kw = dict(w13=q13, w2=q2, w13_scales=c13, w2_scales=c2, shared_w13=a, shared_w13_scales=b, shared_w2=c,
                  shared_w2_scales=d)
    layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, moe.MOE_E4M3 if fp8 else moe.MOE_BF16, **kw)
    bufs = dict(idx=torch.empty(w.T, w.K, dtype=torch.int32, device="cuda"),
                wt=torch.empty(w.T, w.K, dtype=torch.float32, device="cuda"),
                out=torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda"),
                st=torch.zeros(1, dtype=torch.int32, device="cuda"))
    return layer, x, logits, bufs, kw


def test_two_layers_from_two_threads_on_two_streams():
    need_gpu()
    wa = scaled(WORKLOADS["prefill"], T=256, T_valid=256, H=1024, I=512, E=32, K=8)
    wb = scaled(WORKLOADS["decode"], T=128, T_valid=128, H=768, I=256, E=48, K=6)
    la, xa, ga, ba, _ = make(wa, fp8=False)
    lb, xb, gb, bb, _ = make(wb, fp8=True)
    run = lambda l, x, g, b, s: l.forward(x, b["out"], b["idx"], b["wt"], logits=g, dev_status=b["st"], stream=s)
    run(la, xa, ga, ba, None)
    run(lb, xb, gb, bb, None)
    torch.cuda.synchronize()
    want_a, want_b = bits(ba["out"]).copy(), bits(bb["out"]).copy()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    errors = []

    def worker(l, x, g, b, s, want):
        try:
            with torch.cuda.stream(s):
                for _ in range(6):
                    b["out"].zero_()
                    run(l, x, g, b, s)
                    s.synchronize()
                    if not np.array_equal(bits(b["out"]), want):
                        errors.append("mismatch")
        except Exception as e:     # collected and asserted in the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(la, xa, ga, ba, sa, want_a)),
               threading.Thread(target=worker, args=(lb, xb, gb, bb, sb, want_b))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert ba["st"].item() == 0 and bb["st"].item() == 0
