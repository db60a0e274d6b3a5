"""Pins for the oracle's number formats against library routines (torch's CPU casts)
and against the format definitions' special cases."""
import numpy as np
import pytest
import torch

from oracle.formats import (bf16_bits_to_f32, e4m3_decode, e4m3_encode, f32_to_bf16_bits,
                            round_up)


def torch_e4m3_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])


def test_e4m3_encode_matches_torch_on_seeded_values():
    rng = np.random.default_rng(1234)
    n = 2_000_000
    x = (rng.standard_normal(n) * np.exp2(rng.integers(-14, 9, n))).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    assert np.array_equal(e4m3_encode(x), torch_e4m3_bits(x))


def test_e4m3_encode_ties_round_to_even():
    vals = e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)   # 0 .. 448
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)                   # exact halfway points
    assert np.all(mids.astype(np.float64) == (vals[1:] + vals[:-1]) / 2)
    ours = e4m3_encode(mids)
    assert np.array_equal(ours, torch_e4m3_bits(mids))
    # the winner of each tie has an even code (even mantissa)
    assert np.all(ours % 2 == 0)
    assert np.array_equal(e4m3_encode(-mids), ours | 0x80)


def test_e4m3_round_trip_and_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(e4m3_encode(e4m3_decode(codes)), codes)
    big = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, np.inf], np.float32)
    assert np.all(e4m3_encode(big) == 0x7E)
    assert np.all(e4m3_encode(-big) == 0xFE)
    assert e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F
    assert e4m3_encode(np.array([0.0], np.float32))[0] == 0x00
    assert e4m3_encode(np.array([-0.0], np.float32))[0] == 0x80
    # below half the smallest subnormal rounds to zero; exactly half ties to even (0)
    assert e4m3_encode(np.array([2.0 ** -10], np.float32))[0] == 0
    assert e4m3_encode(np.array([2.0 ** -10 * 1.0001], np.float32))[0] == 1


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(99)
    u = rng.integers(0, 2 ** 32, 3_000_000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(f32_to_bf16_bits(x), ref)


def test_bf16_ties_and_overflow():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to the even neighbour 1
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8)], np.float32)
    assert np.array_equal(bf16_bits_to_f32(f32_to_bf16_bits(x)),
                          np.array([1.0, 1 + 2.0 ** -6, -1.0], np.float32))
    biggest = np.float32(np.finfo(np.float32).max)
    assert np.isinf(bf16_bits_to_f32(f32_to_bf16_bits(np.array([biggest])))[0])
    assert f32_to_bf16_bits(np.array([-0.0], np.float32))[0] == 0x8000
    assert np.isnan(bf16_bits_to_f32(f32_to_bf16_bits(np.array([np.nan], np.float32))))[0]


@pytest.mark.parametrize("x,y,r", [(0, 128, 0), (1, 128, 128), (128, 128, 128), (129, 128, 256)])
def test_round_up(x, y, r):
    assert round_up(x, y) == r


def e4m3_encode_by_spacing(x):
    """A second restatement of E4M3 rounding, by value rather than by bit pattern: in
    float64 the spacing of E4M3 values around |x| is 2^-9 below 2^-6, else 2^(e-3) for
    2^e <= |x| < 2^(e+1); |x| / spacing is rounded half to even and scaled back, clamped
    to 448, and the code read off the rounded value."""
    with np.errstate(invalid="ignore"):         # signalling NaN patterns among the inputs
        x = np.asarray(x, dtype=np.float32).astype(np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    _, ex = np.frexp(a)
    e = ex.astype(np.int64) - 1
    step = np.where(a < 2.0 ** -6, 2.0 ** -9, np.exp2(np.maximum(e, -6) - 3.0))
    with np.errstate(invalid="ignore"):         # infinities: inf / step, clamped to 448 below
        v = np.minimum(np.rint(a / step) * step, 448.0)
    _, vex = np.frexp(v)
    ve = vex.astype(np.int64) - 1
    is_sub = v < 2.0 ** -6
    safe_e = np.where(is_sub, 0, ve)
    man = np.rint((v / np.exp2(safe_e) - 1.0) * 8.0).astype(np.int64)
    code = np.where(is_sub, np.rint(v / 2.0 ** -9).astype(np.int64), ((safe_e + 7) << 3) | man)
    code = np.where(nan, 0x7F, code) | np.where(neg, 0x80, 0)
    return code.astype(np.uint8)


def test_e4m3_encode_agrees_with_the_spacing_restatement():
    """Bit-pattern rounding against value rounding: every float32 pattern in [2^-12, 512]
    that lies within 64 ulp of an E4M3 value or of a halfway point between two of them
    (the places where a rounding rule can go wrong), and 4 M random bit patterns."""
    vals = e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    mids = (vals[1:] + vals[:-1]) / 2
    pts = np.concatenate([vals[1:], mids, [464.0, 480.0, 512.0]]).astype(np.float32).view(np.uint32)
    near = (pts[:, None].astype(np.int64) + np.arange(-64, 65)[None, :]).reshape(-1).astype(np.uint32)
    rng = np.random.default_rng(77)
    rand = rng.integers(0, 2 ** 32, 4_000_000, dtype=np.uint64).astype(np.uint32)
    for bitsv in (near, rand):
        x = bitsv.view(np.float32)
        x = np.concatenate([x, -x])
        assert np.array_equal(e4m3_encode(x), e4m3_encode_by_spacing(x))
