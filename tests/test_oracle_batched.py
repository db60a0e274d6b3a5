"""Pins for the oracle's expert-batched permute ([E, max_tokens, H] with per-expert row
counts, the DeepEP page's low-latency format): a case worked by hand from the
definition, its relation to the (separately pinned) contiguous permute when no block
overflows, truncation to the first max_tokens entries of each block, the shared block,
all-padding batches and bad ids."""
import numpy as np
import pytest

from oracle.moe_ref import STATUS_BAD_EXPERT, STATUS_OVERFLOW, permute, permute_batched


def test_worked_example():
    # T=3, K=2, E=3, two rows per block.  Flat slots s = t*K + k:
    #   s: 0 1 2 3 4 5      expert 0 <- s 0, 5; expert 1 <- s 1, 2, 4; expert 2 <- s 3
    #   e: 0 1 1 2 1 0      block 1 keeps s 1, 2 and drops s 4 (its third entry)
    idx = np.array([[0, 1], [1, 2], [1, 0]], dtype=np.int32)
    m, src, inv, smap, st = permute_batched(idx, 3, 2)
    assert m.tolist() == [2, 2, 1]
    assert src.tolist() == [0, 5, 1, 2, 3, -1]
    assert inv.tolist() == [[0, 2], [3, 4], [-1, 1]]
    assert smap is None and st == STATUS_OVERFLOW
    # with the shared block (index 3): every token has a valid slot -> sources 6, 7, 8;
    # two rows per block keep tokens 0 and 1
    m, src, inv, smap, st = permute_batched(idx, 3, 2, with_shared=True)
    assert m.tolist() == [2, 2, 1, 2] and src[6:].tolist() == [6, 7]
    assert smap.tolist() == [6, 7, -1] and st == STATUS_OVERFLOW


def random_idx(T, K, E, pad, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[rng.random((T, K)) < pad] = -1
    return idx


@pytest.mark.parametrize("with_shared", [False, True])
def test_matches_contiguous_layout_without_overflow(with_shared):
    T, K, E = 200, 4, 13
    idx = random_idx(T, K, E, 0.2, seed=1)
    cu, csrc, cinv, csmap, cst = permute(idx, E, with_shared)
    counts = np.diff(cu)
    mt = int(counts.max()) + 3
    m, src, inv, smap, st = permute_batched(idx, E, mt, with_shared)
    assert st == cst == 0
    assert np.array_equal(m, counts)
    for e in range(len(counts)):
        blk = src[e * mt:(e + 1) * mt]
        assert np.array_equal(blk[:counts[e]], csrc[cu[e]:cu[e + 1]])
        assert np.all(blk[counts[e]:] == -1)
    # slot -> row: the contiguous row shifted from its segment start to its block
    seg = np.searchsorted(cu, cinv, side="right") - 1
    want = np.where(cinv >= 0, seg * mt + cinv - cu[np.maximum(seg, 0)], -1)
    assert np.array_equal(inv, want)
    if with_shared:
        sseg = len(counts) - 1
        assert np.array_equal(smap, np.where(csmap >= 0, sseg * mt + csmap - cu[sseg], -1))


def test_overflow_keeps_each_block_prefix():
    T, K, E, mt = 300, 6, 8, 20
    idx = random_idx(T, K, E, 0.1, seed=2)
    cu, csrc, _, _, _ = permute(idx, E)
    m, src, inv, _, st = permute_batched(idx, E, mt)
    assert st == STATUS_OVERFLOW
    assert np.array_equal(m, np.minimum(np.diff(cu), mt))
    for e in range(E):
        assert np.array_equal(src[e * mt:e * mt + m[e]], csrc[cu[e]:cu[e] + m[e]])
    # every kept row maps back to its slot, and dropped slots have no row
    flat = inv.reshape(-1)
    rows = np.nonzero(src >= 0)[0]
    assert np.array_equal(flat[src[rows]], rows)
    assert (flat >= 0).sum() == m.sum()


def test_all_padding_and_bad_ids():
    idx = np.full((5, 3), -1, dtype=np.int32)
    m, src, inv, smap, st = permute_batched(idx, 4, 2, with_shared=True)
    assert m.tolist() == [0] * 5 and np.all(src == -1) and np.all(inv == -1) and np.all(smap == -1) and st == 0
    idx[1, 0], idx[2, 2], idx[3, 1] = 9, -7, 2
    m, src, inv, smap, st = permute_batched(idx, 4, 2, with_shared=True)
    assert st == STATUS_BAD_EXPERT
    assert m.tolist() == [0, 0, 1, 0, 1] and inv[3, 1] == 4 and smap.tolist() == [-1, -1, -1, 8, -1]
