"""Pins for the oracle's permute (counting sort into the expert-major layout): a stable
library sort, the layout's invariants, the shared-expert segment and bad ids."""
import numpy as np
import pytest

from oracle.moe_ref import STATUS_BAD_EXPERT, gather_rows, permute, row_tokens


def random_idx(rng, T, K, E, pad=0.0):
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[rng.random((T, K)) < pad] = -1
    return idx


@pytest.mark.parametrize("T,K,E,pad", [(64, 2, 8, 0.0), (512, 8, 64, 0.1), (100, 4, 32, 0.5),
                                       (7, 3, 3, 0.0)])
def test_matches_stable_library_sort(T, K, E, pad):
    rng = np.random.default_rng(T + K + E)
    idx = random_idx(rng, T, K, E, pad)
    cu, src, inv, _, status = permute(idx, E)
    flat = idx.reshape(-1)
    valid = np.nonzero(flat >= 0)[0]
    order = valid[np.argsort(flat[valid], kind="stable")]     # library stable sort
    N = len(valid)
    assert status == 0
    assert np.array_equal(src[:N], order)
    assert np.all(src[N:] == -1) and len(src) == T * K
    assert np.array_equal(cu, np.concatenate([[0], np.cumsum(np.bincount(flat[valid], minlength=E))]))


@pytest.mark.parametrize("with_shared", [False, True])
def test_invariants(with_shared):
    rng = np.random.default_rng(5)
    T, K, E, H = 300, 6, 40, 16
    idx = random_idx(rng, T, K, E, 0.2)
    idx[17, :] = -1                                   # a padding token
    cu, src, inv, smap, status = permute(idx, E, with_shared=with_shared)
    nseg = E + (1 if with_shared else 0)
    assert len(cu) == nseg + 1 and cu[0] == 0
    assert np.all(np.diff(cu) >= 0)
    n_valid = int((idx >= 0).sum())
    assert cu[E] == n_valid                            # cu_seqlens sums to the valid slots
    flat_inv = inv.reshape(-1)
    # inverse after forward is the identity, both ways
    for p in range(cu[E]):
        assert flat_inv[src[p]] == p
    ok = flat_inv >= 0
    assert np.array_equal(src[flat_inv[ok]], np.nonzero(ok)[0])
    assert np.array_equal(ok, idx.reshape(-1) >= 0)
    # every row of segment e holds a slot routed to e
    for e in range(E):
        assert np.all(idx.reshape(-1)[src[cu[e]:cu[e + 1]]] == e)
    # gather then unpermute returns x repeated
    x = rng.integers(0, 2 ** 16, (T, H), dtype=np.uint16)
    xp = gather_rows(x, src, T, K)
    for s in np.nonzero(ok)[0]:
        assert np.array_equal(xp[flat_inv[s]], x[s // K])
    if with_shared:
        tok_valid = (idx >= 0).any(axis=1)
        assert cu[E + 1] - cu[E] == tok_valid.sum()
        assert np.array_equal(src[cu[E]:cu[E + 1]] - T * K, np.nonzero(tok_valid)[0])
        assert smap[17] == -1
        assert np.array_equal(smap >= 0, tok_valid)
        for t in np.nonzero(tok_valid)[0]:
            assert src[smap[t]] == T * K + t
            assert np.array_equal(xp[smap[t]], x[t])
        assert np.array_equal(row_tokens(src[:cu[-1]], T, K)[cu[E]:], np.nonzero(tok_valid)[0])
    else:
        assert smap is None


def test_bad_ids_are_flagged_and_treated_as_padding():
    idx = np.array([[0, 5], [-2, 1], [1, -1]], np.int32)
    cu, src, inv, _, status = permute(idx, 4)
    assert status & STATUS_BAD_EXPERT
    assert inv[0, 1] == -1 and inv[1, 0] == -1
    assert cu.tolist() == [0, 1, 3, 3, 3]
    assert src[:3].tolist() == [0, 3, 4]


def test_all_padding_batch():
    idx = np.full((8, 4), -1, np.int32)
    cu, src, inv, smap, status = permute(idx, 16, with_shared=True)
    assert status == 0 and np.all(cu == 0)
    assert np.all(src == -1) and np.all(inv == -1) and np.all(smap == -1)
    assert len(src) == 8 * 4 + 8          # capacity from the inputs: T*K (+T)
