"""Pins for the oracle's router (softmax -> top-k -> renormalise): brute force over all
subsets, the closed form of the renormalised weights, tie-breaking and padding rows."""
import itertools
import math

import numpy as np

from oracle.moe_ref import route_topk


def test_topk_set_is_brute_force_argmax():
    rng = np.random.default_rng(7)
    T, E, K = 200, 8, 2
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, w = route_topk(logits, K)
    for t in range(T):
        best = max(itertools.combinations(range(E), K),
                   key=lambda c: sum(float(logits[t, e]) for e in c))
        assert set(idx[t].tolist()) == set(best)
        assert logits[t, idx[t, 0]] >= logits[t, idx[t, 1]]          # descending slot order


def test_weights_closed_form_and_sum():
    rng = np.random.default_rng(8)
    T, E, K = 300, 64, 8
    logits = (rng.standard_normal((T, E)) * 3).astype(np.float32)
    idx, w = route_topk(logits, K)
    for t in range(T):
        # closed form: the full softmax denominator cancels, w_k = e^{l_k} / sum_topk e^{l_j}
        num = [math.exp(float(logits[t, e])) for e in idx[t]]
        ref = np.array([v / sum(num) for v in num], np.float32)
        assert np.max(np.abs(w[t].astype(np.float64) - ref) / ref) <= 2 ** -23
        assert abs(float(w[t].astype(np.float64).sum()) - 1.0) < 1e-6
        assert np.all(np.diff(w[t].astype(np.float64)) <= 0)


def test_ties_go_to_lower_expert_id():
    logits = np.zeros((3, 16), np.float32)
    logits[1, [3, 9, 12]] = 1.0
    idx, w = route_topk(logits, 4)
    assert idx[0].tolist() == [0, 1, 2, 3]
    assert np.allclose(w[0], 0.25)
    assert idx[1].tolist() == [3, 9, 12, 0]
    # -0.0 and +0.0 compare equal: still ordered by id
    logits[2, 5] = -0.0
    assert route_topk(logits[2:3], 2)[0][0].tolist() == [0, 1]


def test_padding_rows_past_num_tokens():
    rng = np.random.default_rng(9)
    logits = rng.standard_normal((10, 8)).astype(np.float32)
    idx, w = route_topk(logits, 2, num_tokens=6)
    assert np.all(idx[6:] == -1) and np.all(w[6:] == 0)
    full_idx, full_w = route_topk(logits, 2)
    assert np.array_equal(idx[:6], full_idx[:6]) and np.array_equal(w[:6], full_w[:6])


def test_k_equals_e_is_sorted_softmax():
    rng = np.random.default_rng(10)
    logits = rng.standard_normal((5, 6)).astype(np.float32)
    idx, w = route_topk(logits, 6)
    for t in range(5):
        assert idx[t].tolist() == list(np.argsort(-logits[t], kind="stable"))
        p = np.exp(logits[t].astype(np.float64))
        p /= p.sum()
        assert np.allclose(w[t], p[idx[t]], rtol=1e-6, atol=0)
