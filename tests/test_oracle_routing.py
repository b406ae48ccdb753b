"""Pins of the oracle's router (top-k + renormalised softmax) and of its stable counting sort.

References used: Python's ``sorted`` on the key (-logit, expert) for the selection and the
tie-break, ``scipy.special.softmax`` for the gates, numpy's stable ``argsort`` / ``bincount``
for the permutation arrays.
"""
import numpy as np
import pytest
from scipy.special import softmax


def _inputs(T, E, seed, ties):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    if ties:
        lg = np.round(lg * 2) / 2          # many exactly equal logits per row
        lg[0, :] = 1.0                      # a row that is all ties
    return lg


@pytest.mark.parametrize("T,E,k,ties", [(16, 8, 2, False), (16, 8, 2, True), (9, 64, 8, True),
                                        (5, 384, 8, False), (4, 384, 8, True), (3, 5, 5, True),
                                        (7, 1, 1, False)])
def test_topk_matches_sorted(oracle_mod, T, E, k, ties):
    lg = _inputs(T, E, T * E + k, ties)
    idx, gate = oracle_mod.route(lg, k)
    for t in range(T):
        ref = sorted(range(E), key=lambda e: (-float(lg[t, e]), e))[:k]
        assert list(idx[t]) == ref
        sm = softmax(lg[t, ref].astype(np.float64))
        np.testing.assert_allclose(gate[t], sm, rtol=1e-13, atol=0)
        assert abs(gate[t].sum() - 1.0) <= 1e-12
        assert np.all(np.diff(gate[t]) <= 0)


def test_all_ties_picks_lowest_indices(oracle_mod):
    lg = np.zeros((2, 16), dtype=np.float32)
    idx, gate = oracle_mod.route(lg, 4)
    assert (idx == np.arange(4)).all()
    assert np.allclose(gate, 0.25, rtol=0, atol=0)


@pytest.mark.parametrize("T,E,k", [(16, 8, 2), (8, 64, 8), (256, 384, 8), (33, 7, 3)])
def test_route_arrays_match_stable_sort(oracle_mod, T, E, k):
    idx, _ = oracle_mod.route(_inputs(T, E, 1, True), k)
    cnt, off, perm, pos = oracle_mod.route_arrays(idx, E)
    flat = idx.ravel()
    assert (cnt == np.bincount(flat, minlength=E)).all()
    assert off[0] == 0 and (off[1:] == np.cumsum(cnt)).all()
    order = np.argsort(flat, kind="stable")          # slot -> flat index t*k + j
    assert (perm == order // k).all()
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    assert (pos == inv).all()
    assert (perm[pos] == np.repeat(np.arange(T), k)).all()
