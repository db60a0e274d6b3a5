"""Pins of the oracle's NVFP4 pieces: the E2M1 element format (value table, nearest-even
rounding against a brute-force search, saturation, signed zero) and the two-level NVFP4
fake-quant of the combine (exact round trips of on-grid blocks, the per-16-element block
scale, the error bound of one element, the zero block, the per-tensor scale) -- none of
them computed by the code they check."""
import numpy as np

from oracle import moe_ref as ref
from oracle.formats import e2m1_decode, e2m1_encode, e2m1_round, e4m3_decode

F32 = np.float32
GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]     # E2M1 magnitudes, codes 0..7


def test_e2m1_value_table_and_round_trip():
    vals = e2m1_decode(np.arange(16))
    assert vals[:8].tolist() == GRID
    assert (-vals[8:]).tolist() == GRID and np.all(np.signbit(vals[8:]))
    assert np.array_equal(e2m1_encode(vals), np.arange(16))


def test_e2m1_ties_and_saturation():
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 6.5, 7.0, 1e30], dtype=F32)
    # each tie goes to the neighbour with an even code: 0(0) 1.0(2) 1.0(2) 2.0(4) 2.0(4) 4.0(6) 4.0(6)
    assert e2m1_round(x).tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, 6.0, 6.0]
    assert e2m1_round(-x).tolist() == [-v for v in [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, 6.0, 6.0]]
    assert np.signbit(e2m1_round(np.array([-0.0, -0.1], dtype=F32))).all()


def test_e2m1_is_the_nearest_grid_value():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-7, 7, 200000), rng.uniform(-1, 1, 50000)]).astype(F32)
    got = e2m1_round(x).astype(np.float64)
    grid = np.array(GRID)
    a = np.abs(x.astype(np.float64))
    d = np.abs(a[:, None] - grid[None, :])
    best = d.min(axis=1)
    assert np.all(np.abs(np.abs(got) - a) == best)         # a nearest magnitude
    # ties (two nearest values) take the even code; away from ties the nearest is unique
    n_near = (d == best[:, None]).sum(axis=1)
    codes = e2m1_encode(x) & 7
    assert np.all((codes[n_near == 2] & 1) == 0)
    assert np.all(np.sign(got[got != 0]) == np.sign(x[got != 0]))


def on_grid_rows(rng, rows, blocks, exps):
    """Rows whose 16-element blocks are E2M1 values times 2^e with one block element at
    magnitude 6 (so the block's amax is 6 * 2^e)."""
    v = rng.choice(np.array(GRID), size=(rows, blocks, 16)) * rng.choice([-1.0, 1.0], size=(rows, blocks, 16))
    v[:, :, 0] = 6.0
    return (v * np.exp2(np.asarray(exps, dtype=np.float64))[None, :, None]).reshape(rows, blocks * 16).astype(F32)


def test_nvfp4_round_trip_of_on_grid_blocks_is_exact():
    # g = 1 (calibration amax 2688): block scale = amax / 6 = 2^e, an E4M3 value; every
    # element is an exact E2M1 multiple of it, so the fake-quant returns the row unchanged.
    # Per-block exponents differ, which a wrong block size (e.g. 32) would not survive.
    rng = np.random.default_rng(2)
    r = on_grid_rows(rng, 5, 8, [0, 3, -2, 5, 1, -4, 2, 0])
    g = ref.nvfp4_scale_from_amax(F32(2688.0))
    assert g == F32(1.0)
    assert np.array_equal(ref.nvfp4_qdq_f32(r, g), r)
    # the same with a power-of-two per-tensor scale: still exact
    assert np.array_equal(ref.nvfp4_qdq_f32(r, F32(4.0)), r)


def test_nvfp4_block_scale_and_element_error_bound():
    rng = np.random.default_rng(3)
    r = (rng.standard_normal((64, 256)) * rng.uniform(0.01, 10, (64, 1))).astype(F32)
    amax = F32(np.abs(r).max())
    g = ref.nvfp4_scale_from_amax(amax)
    assert g == F32(F32(2688.0) / amax)
    q = ref.nvfp4_qdq_f32(r, g)
    blocks = r.reshape(64, 16, 16).astype(np.float64)
    qb = q.reshape(64, 16, 16).astype(np.float64)
    a = np.abs(blocks).max(axis=2, keepdims=True)
    # each block's dequantisation step d is its E4M3-rounded scale over g; elements land on
    # E2M1 multiples of d, at most 6 d in magnitude
    sf = ((a.astype(F32) / F32(6.0)).astype(F32) * g).astype(F32)
    from oracle.formats import e4m3_encode
    d = (e4m3_decode(e4m3_encode(sf)) / g).astype(np.float64)
    ratio = qb / d
    assert np.all(np.isin(np.abs(np.round(ratio, 6)), GRID))
    # an element is off by at most half the E2M1 spacing at its magnitude (1 * d at most),
    # plus the float32 roundings of the scaled value and the product
    assert np.all(np.abs(qb - blocks) <= d * 1.0 + 1e-6 * np.abs(blocks) + 1e-30)
    # the largest element of a block keeps its magnitude within that bound and its sign
    assert np.all(np.sign(qb[np.abs(qb) > 0]) == np.sign(blocks[np.abs(qb) > 0]))


def test_nvfp4_zero_block_and_scale_of_zero_amax():
    r = np.zeros((2, 32), dtype=F32)
    r[1, 16:] = np.linspace(-1, 1, 16, dtype=F32)
    q = ref.nvfp4_qdq_f32(r, F32(3.0))
    assert np.all(q[0] == 0) and np.all(q[1, :16] == 0)
    assert ref.nvfp4_scale_from_amax(F32(0.0)) == F32(1.0)


def test_combine_with_nvfp4_on_grid_rows_equals_the_plain_combine():
    """Weights 1 and on-grid rows: the NVFP4 fake-quant changes nothing, so the combine's
    result is the plain one; off-grid rows change it."""
    rng = np.random.default_rng(4)
    T, K, H = 6, 3, 64
    y = on_grid_rows(rng, T * K, H // 16, [0, 1, -1, 2])
    from oracle.formats import f32_to_bf16_bits
    yb = f32_to_bf16_bits(y)
    inv = np.arange(T * K, dtype=np.int32).reshape(T, K)
    inv[2, 1] = -1
    w = np.ones((T, K), dtype=F32)
    g = F32(1.0)
    assert np.array_equal(ref.combine(yb, inv, w, fq_scale=g, fq_format="nvfp4"), ref.combine(yb, inv, w))
    yo = f32_to_bf16_bits((y * F32(1.1)).astype(F32))
    assert not np.array_equal(ref.combine(yo, inv, w, fq_scale=g, fq_format="nvfp4"), ref.combine(yo, inv, w))


def test_nvfp4_dispatch_fake_quant_of_bf16_rows():
    """Dispatch (the page's other NVFP4 unit): on-grid BF16 rows come back unchanged at
    g = 1; off-grid rows land on the block grids and are rounded to BF16; the E4M3 default
    is untouched by the format argument."""
    from oracle.formats import bf16_bits_to_f32, f32_to_bf16_bits
    rng = np.random.default_rng(6)
    r = on_grid_rows(rng, 4, 8, [0, 2, -3, 1, 4, -1, 0, 3])
    rb = f32_to_bf16_bits(r)
    assert np.array_equal(ref.dispatch_qdq_bits(rb, F32(1.0), "nvfp4"), rb)
    x = f32_to_bf16_bits((rng.standard_normal((4, 128)) * 2).astype(F32))
    g = ref.nvfp4_scale_from_amax(ref.tensor_amax(x))
    got = ref.dispatch_qdq_bits(x, g, "nvfp4")
    assert np.array_equal(got, f32_to_bf16_bits(ref.nvfp4_qdq_f32(bf16_bits_to_f32(x), g)))
    assert not np.array_equal(got, x)
    assert np.array_equal(ref.dispatch_qdq_bits(x, F32(7.0)), ref.dispatch_qdq_bits(x, F32(7.0), "e4m3"))
