"""Pins for the oracle's FP8 block quantisers (1x128 activations, 128x128 weights):
block maxima land on +-448, reconstruction within half an E4M3 step, the rounding step
equal to torch's cast of the float32 quotient, and all-zero blocks."""
import numpy as np
import torch

from oracle.formats import e4m3_decode
from oracle.moe_ref import act_quant_1x128, dequant, weight_quant_128x128


def torch_cast(v):
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def check_blocks(x, q, s, br):
    R, C = x.shape
    xb = x.reshape(R // br, br, C // 128, 128)
    qb = q.reshape(R // br, br, C // 128, 128)
    amax = np.abs(xb).max(axis=(1, 3))
    assert np.array_equal(s, np.where(amax > 0, (amax / np.float32(448)).astype(np.float32), 1))
    # the rounding step is torch's cast of the float32 quotient x / s (|x / s| <= 448 here)
    quo = (xb / s[:, None, :, None]).astype(np.float32)
    assert np.abs(quo).max() <= 448.0 * (1 + 2.0 ** -22)
    assert np.array_equal(qb[np.abs(quo) <= 448], torch_cast(quo[np.abs(quo) <= 448]))
    # each nonzero block's largest magnitude encodes to +-448 (code 0x7E / 0xFE)
    for i in range(R // br):
        for j in range(C // 128):
            blk = xb[i, :, j, :]
            if amax[i, j] > 0:
                pos = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
                assert qb[i, pos[0], j, pos[1]] & 0x7F == 0x7E
    # reconstruction within half an E4M3 step (relative 2^-4), or the subnormal step
    rec = dequant(q, s, br)
    srep = np.repeat(np.repeat(s.astype(np.float64), br, 0), 128, 1)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, srep * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(rec - x) <= bound)


def test_act_quant_1x128():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((40, 512)) * np.exp2(rng.integers(-6, 6, (40, 1)))).astype(np.float32)
    x[3, 128:256] = 0.0
    q, s = act_quant_1x128(x)
    assert q.shape == x.shape and s.shape == (40, 4)
    assert s[3, 1] == 1.0 and np.all(q[3, 128:256] == 0)
    check_blocks(x, q, s, 1)


def test_weight_quant_128x128():
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((256, 384)) * 0.02).astype(np.float32)
    w[128:, :128] = 0.0
    q, s = weight_quant_128x128(w)
    assert s.shape == (2, 3) and s[1, 0] == 1.0
    check_blocks(w, q, s, 128)


def test_exactly_representable_block_is_lossless():
    codes = np.arange(0, 126, dtype=np.uint8)        # 0 .. 448, all finite positives
    v = e4m3_decode(np.concatenate([codes, [0x7E, 0x7E]]))[:128] * np.float32(0.25)
    x = np.stack([v, -v]).astype(np.float32)
    q, s = act_quant_1x128(x)
    assert np.all(s == np.float32(112.0 / 448.0))
    assert np.array_equal(dequant(q, s, 1), x.astype(np.float64))
