"""Pins of the oracle's rejection-sampling verification of a drafted block.

Statistical pins (the closed forms of speculative sampling): with drafted tokens drawn from
q, a position is accepted with probability sum_x min(p(x), q(x)) and the first emitted token
is distributed as p (the method is lossless).  Exact pins: the fixed-point inverse-CDF draw
against a numpy cumulative sum of the same integer masses, and edge cases whose outcome is
forced (p == q accepts everything; p(d) = 0 < q(d) rejects; the residual's support).
"""
import numpy as np
import pytest

from oracle import oracle as O


def _draw_ref(w, U):
    """first x with cumsum(floor(w * 2^62)) > floor(U * M / 2^64), in Python integers"""
    m = [int(np.floor(float(v) * 2.0 ** 62)) for v in w]
    M = sum(m)
    if M == 0:
        return -1
    t = (int(U) * M) >> 64
    run = 0
    for x, mx in enumerate(m):
        run += mx
        if run > t:
            return x
    raise AssertionError


def _one_position(p0, q0, p1, d, u, U):
    """verify a single drafted token (g = 1)"""
    S = len(d)
    p = np.stack([np.broadcast_to(p0, (S, p0.size)), np.broadcast_to(p1, (S, p1.size))], axis=1)
    q = np.broadcast_to(q0, (S, 1, q0.size))
    return O.verify(p, q, d.reshape(S, 1), u.reshape(S, 1), U)


def test_acceptance_rate_is_one_minus_total_variation():
    rng = np.random.default_rng(1)
    V = 6
    p = np.array([0.30, 0.25, 0.20, 0.15, 0.07, 0.03], np.float32)
    q = np.array([0.10, 0.10, 0.35, 0.15, 0.20, 0.10], np.float32)
    S = 200000
    d = rng.choice(V, size=S, p=q / q.sum()).astype(np.int32)
    u = (rng.integers(0, 2 ** 24, size=S) / 2.0 ** 24).astype(np.float32)
    U = rng.integers(0, 2 ** 64, size=S, dtype=np.uint64)
    n_acc, tok = _one_position(p, q, p, d, u, U)
    rate = n_acc.mean()
    want = float(np.minimum(p.astype(np.float64), q.astype(np.float64)).sum())
    assert abs(rate - want) < 4 * np.sqrt(want * (1 - want) / S)
    # lossless: the first emitted token (accepted draft or residual draw) follows p
    first = tok[:, 0]
    counts = np.bincount(first, minlength=V)
    expected = S * p.astype(np.float64) / p.sum()
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 25.0                                     # 5 dof: p-value ~ 1e-4


def test_equal_distributions_accept_everything_then_draw_bonus():
    rng = np.random.default_rng(2)
    S, g, V = 50, 7, 40
    p = rng.dirichlet(np.ones(V), size=(S, g + 1)).astype(np.float32)
    q = p[:, :g].copy()
    d = rng.integers(0, V, (S, g)).astype(np.int32)
    d[0, 3] = int(np.argmax(p[0, 3]))
    u = (rng.integers(0, 2 ** 24, (S, g)) / 2.0 ** 24).astype(np.float32)
    U = rng.integers(0, 2 ** 64, S, dtype=np.uint64)
    n_acc, tok = O.verify(p, q, d, u, U)
    assert (n_acc == g).all()
    assert (tok[:, :g] == d).all()
    for s in range(S):
        assert tok[s, g] == _draw_ref(p[s, g], U[s])


def test_zero_target_probability_rejects_and_residual_support():
    S, g, V = 4, 3, 8
    p = np.full((S, g + 1, V), 1.0 / V, np.float32)
    q = np.full((S, g, V), 1.0 / V, np.float32)
    p[:, 1, 5] = 0.0                                       # draft 5 impossible at position 1
    p[:, 1, 2] += 1.0 / V                                  # the residual is all on token 2
    d = np.zeros((S, g), np.int32)
    d[:, 1] = 5
    u = np.zeros((S, g), np.float32)
    U = np.array([0, 1, 2 ** 63, 2 ** 64 - 1], np.uint64)
    n_acc, tok = O.verify(p, q, d, u, U)
    assert (n_acc == 1).all()
    assert (tok[:, 0] == 0).all() and (tok[:, 1] == 2).all() and (tok[:, 2:] == -1).all()


@pytest.mark.parametrize("seed", [3, 4])
def test_fixed_point_draw_matches_integer_cumsum(seed):
    rng = np.random.default_rng(seed)
    S, g, V = 64, 2, 257
    p = rng.dirichlet(np.full(V, 0.3), size=(S, g + 1)).astype(np.float32)
    q = rng.dirichlet(np.full(V, 0.3), size=(S, g)).astype(np.float32)
    d = rng.integers(0, V, (S, g)).astype(np.int32)
    u = (rng.integers(0, 2 ** 24, (S, g)) / 2.0 ** 24).astype(np.float32)
    U = rng.integers(0, 2 ** 64, S, dtype=np.uint64)
    U[:3] = [0, 2 ** 64 - 1, 2 ** 32]
    n_acc, tok = O.verify(p, q, d, u, U)
    for s in range(S):
        i = int(n_acc[s])
        for j in range(i):                                 # accepted: u q(d) < p(d) exactly
            assert float(u[s, j]) * float(q[s, j, d[s, j]]) < float(p[s, j, d[s, j]])
            assert tok[s, j] == d[s, j]
        if i < g:
            assert float(u[s, i]) * float(q[s, i, d[s, i]]) >= float(p[s, i, d[s, i]])
            r = np.maximum(p[s, i] - q[s, i], np.float32(0))   # fp32 difference
            want = _draw_ref(r, U[s])
        else:
            want = _draw_ref(p[s, g], U[s])
        assert tok[s, i] == want
        assert (tok[s, i + 1:] == -1).all()


def test_verify_rejects_bad_arguments():
    p = np.full((1, 2, 4), 0.25, np.float32)
    q = np.full((1, 1, 4), 0.25, np.float32)
    with pytest.raises(ValueError):
        O.verify(p, q, np.array([[7]], np.int32), np.zeros((1, 1), np.float32),
                 np.zeros(1, np.uint64))
