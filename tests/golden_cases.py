"""Loader for the hand-derived combine fixtures in tests/golden/combine_order.json.

Each case becomes one token's combine problem: the rows of its valid slots in an
expert-output buffer Y (plus one garbage row that padding slots must never read), an
inverse map, router weights and an optional shared row.
"""
import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
H = 256   # each case's value is repeated over H columns (several 16-byte vectors)


def _f32_bits_to_bf16(v):
    b = np.array([v], np.float32).view(np.uint32)[0] >> 16
    assert (np.array([v], np.float32).view(np.uint32)[0] & 0xFFFF) == 0, "not exact in BF16"
    return np.uint16(b)


def load_cases():
    with open(os.path.join(HERE, "golden", "combine_order.json")) as f:
        return json.load(f)["cases"]


def build(case):
    """-> dict(y [R, H] uint16, inv_map [1, K] int32, w [1, K] float32,
    shared [1, H] uint16 | None, fq_scale float | None, expect uint16)."""
    rows = case["rows"]
    K = len(rows)
    garbage = np.uint16(0x7F7F)                   # largest finite BF16, about 3.4e38
    y = [np.full(H, garbage, np.uint16)]          # row 0: garbage, never referenced
    inv = []
    for r in rows:
        if r is None:
            inv.append(-1)
        else:
            y.append(np.full(H, _f32_bits_to_bf16(np.float32(float.fromhex(r))), np.uint16))
            inv.append(len(y) - 1)
    w = np.array([[float.fromhex(v) for v in case["w"]]], np.float32)
    shared = None
    if case["shared"] is not None:
        shared = np.full((1, H), _f32_bits_to_bf16(np.float32(float.fromhex(case["shared"]))),
                         np.uint16)
    fq = None if case["fq_scale"] is None else float.fromhex(case["fq_scale"])
    return dict(y=np.stack(y), inv_map=np.array([inv], np.int32), w=w, shared=shared,
                fq_scale=fq, expect=np.uint16(int(case["expect_bits"], 16)), K=K)
