"""Pins for the oracle's fixed-order combine and its fake-quant: hand-derived golden
cases (tests/golden/combine_order.json), the identity-expert closed form out = K * x,
padding semantics and the calibration amax."""
import numpy as np
import pytest

from golden_cases import build, load_cases
from oracle.formats import bf16_bits_to_f32, e4m3_decode, f32_to_bf16_bits
from oracle.moe_ref import (combine, combine_amax, fq_scale_from_amax, gather_rows, permute,
                            qdq_f32)


@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c["name"])
def test_golden_case(case):
    c = build(case)
    out = combine(c["y"], c["inv_map"], c["w"], shared_bits=c["shared"], fq_scale=c["fq_scale"])
    assert out.shape == (1, c["y"].shape[1])
    assert np.all(out == c["expect"]), (hex(out[0, 0]), hex(c["expect"]))


@pytest.mark.parametrize("K", [1, 2, 3, 8])
def test_identity_experts_give_k_times_x(K):
    """All router weights 1 and identity experts (each row = the token's x): the
    combine returns bf16(K * x).  Partial sums j*x (j <= 8) of a BF16 x are exact in
    float32, so only the final rounding acts -- for K = 1, 2, 8 that is exact too."""
    rng = np.random.default_rng(K)
    T, H, E = 37, 384, 9
    x = f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    cu, src, inv, _, _ = permute(idx, E)
    y = gather_rows(x, src, T, K)                       # identity experts
    out = combine(y, inv, np.ones((T, K), np.float32))
    kx = (bf16_bits_to_f32(x) * np.float32(K)).astype(np.float32)
    assert np.array_equal(out, f32_to_bf16_bits(kx))
    if K in (1, 2, 8):
        assert np.array_equal(bf16_bits_to_f32(out), kx)


def test_padding_slots_and_tokens():
    rng = np.random.default_rng(3)
    T, H, E, K = 16, 128, 4, 3
    x = f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[2, 1] = -1
    idx[5, :] = -1
    cu, src, inv, smap, _ = permute(idx, E, with_shared=True)
    y = gather_rows(x, src, T, K)
    w = np.ones((T, K), np.float32)
    out = combine(y, inv, w, shared_bits=y, shared_map=smap)
    assert np.all(out[5] == 0)                           # padding token: +0, no shared row
    kx2 = (bf16_bits_to_f32(x[2]) * np.float32(2) + bf16_bits_to_f32(x[2])).astype(np.float32)
    assert np.array_equal(out[2], f32_to_bf16_bits(kx2))  # 2 valid slots + shared
    # dense shared rows give the same result as the mapped ones
    assert np.array_equal(out, combine(y, inv, w, shared_bits=x))


def test_qdq_exact_values_pass_through():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    v = e4m3_decode(codes)
    for s in (1.0, 2.0 ** 5, 2.0 ** -3):
        r = (v / np.float32(s)).astype(np.float32)         # exact: s is a power of two
        assert np.array_equal(qdq_f32(r, s), r)


def test_qdq_saturates_and_rounds():
    s = np.float32(448.0 / 3.0)
    r = np.array([3.0, -3.0, 30.0], np.float32)
    out = qdq_f32(r, s)
    assert out[2] == np.float32(np.float32(448.0) / s)
    assert out[0] == -out[1]
    # relative error of a normal-range value is at most half an E4M3 step (2^-4)
    rng = np.random.default_rng(5)
    r = rng.uniform(-3, 3, 100000).astype(np.float32)
    q = qdq_f32(r, s)
    big = np.abs(r * s) >= 2.0 ** -6
    assert np.all(np.abs(q[big] - r[big]) <= np.abs(r[big]) * 2.0 ** -4 * 1.0001)


def test_calibration_amax_and_scale():
    rng = np.random.default_rng(11)
    T, H, E, K = 20, 128, 6, 2
    x = f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[3, 0] = -1
    w = rng.uniform(0.1, 1.0, (T, K)).astype(np.float32)
    cu, src, inv, _, _ = permute(idx, E)
    y = gather_rows(x, src, T, K)
    xf = bf16_bits_to_f32(x)
    brute = 0.0
    for t in range(T):
        for k in range(K):
            if idx[t, k] >= 0:
                brute = max(brute, float(np.abs((xf[t] * w[t, k]).astype(np.float32)).max()))
    amax = combine_amax(y, inv, w)
    assert amax == np.float32(brute)
    s = fq_scale_from_amax(amax)
    assert s == np.float32(np.float32(448.0) / np.float32(brute))
    # the largest weighted row element maps to (about) the E4M3 maximum
    assert abs(float(np.float32(amax) * s) - 448.0) <= 448.0 * 2.0 ** -23
    assert fq_scale_from_amax(0.0) == 1.0


def test_dispatch_qdq_pins():
    from oracle.moe_ref import dispatch_qdq_bits, tensor_amax
    # exactly representable E4M3 values (times a power-of-two scale) pass through
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    v = e4m3_decode(codes) / np.float32(8.0)
    bits = f32_to_bf16_bits(v)
    assert np.array_equal(dispatch_qdq_bits(bits, 8.0), bits)
    # the rounding step is torch's E4M3 cast of the float32 product (library routine)
    import torch
    rng = np.random.default_rng(21)
    x = f32_to_bf16_bits(rng.standard_normal(50000).astype(np.float32))
    s = np.float32(448.0) / tensor_amax(x)
    xf = bf16_bits_to_f32(x)
    t = (xf * s).astype(np.float32)
    q = torch.from_numpy(t).to(torch.float8_e4m3fn).float().numpy()
    want = f32_to_bf16_bits((q / s).astype(np.float32))
    assert np.array_equal(dispatch_qdq_bits(x, s), want)
    assert tensor_amax(x) == np.abs(xf).max()


def test_preweighted_rows_equal_unit_weights():
    """Rows already router-weighted (topk_w None) reduce to the weighted combine with all
    weights 1, since float32(y * 1) = y exactly; with fake-quant too."""
    rng = np.random.default_rng(31)
    T, H, E, K = 40, 256, 12, 4
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[rng.random((T, K)) < 0.2] = -1
    cu, src, inv, smap, _ = permute(idx, E, with_shared=True)
    y = f32_to_bf16_bits(rng.standard_normal((len(src), H)).astype(np.float32))
    ones = np.ones((T, K), np.float32)
    for fq in (None, 96.0):
        a = combine(y, inv, None, shared_bits=y, shared_map=smap, fq_scale=fq)
        b = combine(y, inv, ones, shared_bits=y, shared_map=smap, fq_scale=fq)
        assert np.array_equal(a, b)
    assert combine_amax(y, inv, None) == combine_amax(y, inv, ones)
