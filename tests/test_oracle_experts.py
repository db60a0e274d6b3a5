"""Pins for the oracle's SwiGLU experts and the dense per-token layer reference:
brute-force scalar loops on tiny inputs, the silu odd-part identity (catches a sign
error or swapped gate/up halves), and the FP8 reference against the BF16 one."""
import math

import numpy as np
import pytest

from oracle.formats import bf16_bits_to_f32, f32_to_bf16_bits
from oracle.moe_ref import layer_reference, max_rel_err, route_topk, swiglu_expert


def brute_expert(x, w13, w2):
    """Scalar loops: y_j = sum_i W2[j, i] * silu(sum_h Wg[i, h] x_h) * (sum_h Wu[i, h] x_h)."""
    I = len(w13) // 2
    H = len(x)
    h = []
    for i in range(I):
        g = sum(float(w13[i][c]) * float(x[c]) for c in range(H))
        u = sum(float(w13[I + i][c]) * float(x[c]) for c in range(H))
        h.append(g / (1.0 + math.exp(-g)) * u)
    return [sum(float(w2[j][i]) * h[i] for i in range(I)) for j in range(len(w2))]


def test_expert_matches_scalar_loops():
    rng = np.random.default_rng(1)
    H, I = 7, 5
    x = rng.standard_normal((3, H))
    w13 = rng.standard_normal((2 * I, H))
    w2 = rng.standard_normal((H, I))
    y = swiglu_expert(x, w13, w2)
    for m in range(3):
        assert np.allclose(y[m], brute_expert(x[m], w13, w2), rtol=1e-12, atol=1e-12)


def test_silu_odd_part_identity():
    """silu(g) - silu(-g) = g, so negating the gate rows changes the output by
    W_down (g * u): a bilinear form with no silu in it."""
    rng = np.random.default_rng(2)
    H, I = 32, 24
    x = rng.standard_normal((10, H))
    w13 = rng.standard_normal((2 * I, H))
    w2 = rng.standard_normal((H, I))
    neg = w13.copy()
    neg[:I] *= -1
    g = x @ w13[:I].T
    u = x @ w13[I:].T
    diff = swiglu_expert(x, w13, w2) - swiglu_expert(x, neg, w2)
    assert np.allclose(diff, (g * u) @ w2.T, rtol=1e-10, atol=1e-10)


def brute_layer(x, idx, w, w13, w2, shared):
    T, K = idx.shape
    out = np.zeros((T, x.shape[1]))
    for t in range(T):
        acc = [0.0] * x.shape[1]
        any_valid = False
        for k in range(K):
            e = idx[t, k]
            if e < 0:
                continue
            any_valid = True
            y = brute_expert(x[t], w13[e], w2[e])
            acc = [a + float(w[t, k]) * b for a, b in zip(acc, y)]
        if any_valid and shared is not None:
            y = brute_expert(x[t], shared[0], shared[1])
            acc = [a + b for a, b in zip(acc, y)]
        out[t] = acc
    return out


@pytest.mark.parametrize("with_shared", [False, True])
def test_layer_reference_matches_brute_force(with_shared):
    rng = np.random.default_rng(3)
    T, H, I, E, K = 9, 6, 4, 5, 2
    xb = f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    idx, w = route_topk(rng.standard_normal((T, E)).astype(np.float32), K)
    idx[4, 1] = -1
    idx[6, :] = -1
    w13 = f32_to_bf16_bits(rng.standard_normal((E, 2 * I, H)).astype(np.float32))
    w2 = f32_to_bf16_bits(rng.standard_normal((E, H, I)).astype(np.float32))
    shared = None
    if with_shared:
        shared = (f32_to_bf16_bits(rng.standard_normal((2 * I, H)).astype(np.float32)),
                  f32_to_bf16_bits(rng.standard_normal((H, I)).astype(np.float32)))
    ref = layer_reference(xb, idx, w, w13, w2, shared=shared)
    f = lambda a: bf16_bits_to_f32(a).astype(np.float64)
    brute = brute_layer(f(xb), idx, w, f(w13), f(w2),
                        None if shared is None else (f(shared[0]), f(shared[1])))
    assert np.allclose(ref, brute, rtol=1e-12, atol=1e-12)
    assert np.all(ref[6] == 0)
    # a token subset gives the same rows
    sub = layer_reference(xb, idx, w, w13, w2, shared=shared, tokens=[8, 2, 4])
    assert np.allclose(sub, ref[[8, 2, 4]], rtol=1e-12, atol=1e-12)


def test_fp8_reference_error_is_the_fp8_rounding_error():
    """The FP8 reference differs from the BF16 one by E4M3's own rounding error: four
    quantised operands (x, W13, h, W2), each with a uniform relative rounding error of
    rms 2^-4/sqrt(3) = 3.6%, give about sqrt(4) * 3.6% = 7% rms on the output."""
    rng = np.random.default_rng(4)
    T, H, I, E, K = 16, 256, 256, 4, 2
    xb = f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    idx, w = route_topk(rng.random((T, E)).astype(np.float32), K)
    w13 = f32_to_bf16_bits((rng.standard_normal((E, 2 * I, H)) / math.sqrt(H)).astype(np.float32))
    w2 = f32_to_bf16_bits((rng.standard_normal((E, H, I)) / math.sqrt(I)).astype(np.float32))
    ref = layer_reference(xb, idx, w, w13, w2)
    ref8 = layer_reference(xb, idx, w, w13, w2, fp8=True)
    rms = np.sqrt(((ref8 - ref) ** 2).mean() / (ref ** 2).mean())
    assert 0.03 < rms < 0.10
    assert max_rel_err(ref8, ref) < 0.15


def test_layer_reference_dispatch_fake_quant_routes_quantised_tokens_only():
    """Routed experts see the fake-quantised tokens, the shared expert the original ones."""
    from oracle.moe_ref import dispatch_qdq_bits
    rng = np.random.default_rng(5)
    T, H, I, E, K = 7, 6, 4, 5, 2
    xb = f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    idx, w = route_topk(rng.standard_normal((T, E)).astype(np.float32), K)
    w13 = f32_to_bf16_bits(rng.standard_normal((E, 2 * I, H)).astype(np.float32))
    w2 = f32_to_bf16_bits(rng.standard_normal((E, H, I)).astype(np.float32))
    shared = (f32_to_bf16_bits(rng.standard_normal((2 * I, H)).astype(np.float32)),
              f32_to_bf16_bits(rng.standard_normal((H, I)).astype(np.float32)))
    s = np.float32(20.0)
    ref = layer_reference(xb, idx, w, w13, w2, shared=shared, dispatch_scale=s)
    f = lambda a: bf16_bits_to_f32(a).astype(np.float64)
    routed_only = brute_layer(f(dispatch_qdq_bits(xb, s)), idx, w, f(w13), f(w2), None)
    shared_only = np.stack([brute_expert(f(xb)[t], f(shared[0]), f(shared[1])) for t in range(T)])
    assert np.allclose(ref, routed_only + shared_only, rtol=1e-12, atol=1e-12)
    assert not np.allclose(ref, layer_reference(xb, idx, w, w13, w2, shared=shared), rtol=1e-3, atol=0)


# ------------------------------------------------------------------ FP8 branch, by loops
def _e4m3_value(v):
    """E4M3 rounding of one float32 value through torch's cast (a library routine, round
    to nearest even), saturating at +-448 by the format's definition (e4m3fn has no inf)."""
    import torch
    v = max(-448.0, min(448.0, float(np.float32(v))))
    return float(torch.tensor([v], dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float32).item())


def _block_quant_loops(m, block_rows):
    """Dequantised FP8 blocks of a float32 matrix, element by element: per block of
    block_rows x 128, s = fl32(amax / 448) (1 for an all-zero block), each element
    e4m3(fl32(v / s)) * s (the float32 division of the FP8 path, then fp64)."""
    m = np.asarray(m, dtype=np.float32)
    R, C = m.shape
    out = np.zeros((R, C))
    for r0 in range(0, R, block_rows):
        for c0 in range(0, C, 128):
            amax = 0.0
            for r in range(r0, r0 + block_rows):
                for c in range(c0, c0 + 128):
                    amax = max(amax, abs(float(m[r, c])))
            s = np.float32(np.float32(amax) / np.float32(448.0))
            s = s if s > 0 else np.float32(1.0)
            for r in range(r0, r0 + block_rows):
                for c in range(c0, c0 + 128):
                    out[r, c] = _e4m3_value(np.float32(m[r, c] / s)) * float(s)
    return out


def _fp8_expert_loops(x_row, w13, w2):
    """One FP8 expert on one token, every step from its definition: x quantised per 1x128
    block, W13 and W2 per 128x128 block, g and u as plain dot products, h = silu(g) * u
    rounded to float32 and re-quantised per 1x128 block, then the down product."""
    I = w13.shape[0] // 2
    xq = _block_quant_loops(x_row[None, :], 1)[0]
    w13q = _block_quant_loops(w13, 128)
    w2q = _block_quant_loops(w2, 128)
    h = np.zeros(I, dtype=np.float32)
    for i in range(I):
        g = math.fsum(w13q[i, c] * xq[c] for c in range(len(xq)))
        u = math.fsum(w13q[I + i, c] * xq[c] for c in range(len(xq)))
        h[i] = np.float32(g / (1.0 + math.exp(-g)) * u)
    hq = _block_quant_loops(h[None, :], 1)[0]
    return np.array([math.fsum(w2q[j, i] * hq[i] for i in range(I)) for j in range(w2.shape[0])]), h


def test_fp8_layer_reference_matches_scalar_loops():
    """The FP8 branch of the layer reference (x and h quantised per 1x128 block, weights per
    128x128 block, the SwiGLU output re-quantised before the down projection) against
    the same expert computed element by element, on routed slots and a shared expert with
    H = I = 256 (two blocks along every axis).  A reference that skipped the re-quantisation
    of h, or quantised h with one scale per 128 x 128 block, would differ by E4M3's rounding
    error (percent level); the two checks at the end show this case tells them apart."""
    rng = np.random.default_rng(6)
    T, H, I, E, K = 3, 256, 256, 2, 2
    xb = f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    idx, w = route_topk(rng.standard_normal((T, E)).astype(np.float32), K)
    idx[2, 1] = -1
    w13 = f32_to_bf16_bits((rng.standard_normal((E, 2 * I, H)) / 16).astype(np.float32))
    w2 = f32_to_bf16_bits((rng.standard_normal((E, H, I)) / 16).astype(np.float32))
    shared = (f32_to_bf16_bits((rng.standard_normal((2 * I, H)) / 16).astype(np.float32)),
              f32_to_bf16_bits((rng.standard_normal((H, I)) / 16).astype(np.float32)))
    ref8 = layer_reference(xb, idx, w, w13, w2, shared=shared, fp8=True)
    f = lambda a: bf16_bits_to_f32(a)
    x = f(xb)
    want = np.zeros((T, H))
    hs = []
    for t in range(T):
        for k in range(K):
            if idx[t, k] < 0:
                continue
            y, h = _fp8_expert_loops(x[t], f(w13[idx[t, k]]), f(w2[idx[t, k]]))
            want[t] += float(w[t, k]) * y
            hs.append((h, f(w2[idx[t, k]])))
        ys, _ = _fp8_expert_loops(x[t], f(shared[0]), f(shared[1]))
        want[t] += ys
    scale = np.abs(want).max()
    assert np.allclose(ref8, want, rtol=1e-9, atol=1e-12 * scale)
    # sensitivity: the down product of an un-requantised h, or of h quantised with a scale
    # shared by the rows of a 128 x 128 block, moves the output far outside that bound
    h, w2e = hs[0]
    w2q = _block_quant_loops(w2e, 128)
    per_row = w2q @ _block_quant_loops(h[None, :], 1)[0]
    plain = w2q @ h.astype(np.float64)
    h2 = np.stack([h, 3.7 * h])                      # a second row with a larger amax
    shared_block = w2q @ _block_quant_loops(np.pad(h2, ((0, 126), (0, 0))), 128)[0]
    assert np.abs(plain - per_row).max() > 1e-4 * np.abs(per_row).max()
    assert np.abs(shared_block - per_row).max() > 1e-4 * np.abs(per_row).max()
