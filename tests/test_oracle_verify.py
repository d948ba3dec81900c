"""Pins of the rejection-sampling verifier oracle (no GPU): the hand-worked
cases, brute-force integration of the method's guarantee (the output token
follows the target distribution exactly, whatever the draft distribution),
and special cases."""

import os

import numpy as np

from oracle import verify as ov

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
P_T = np.array([[0.1, 0.4, 0.3, 0.2], [0.25, 0.25, 0.25, 0.25]])
P_D = np.array([[0.4, 0.2, 0.2, 0.2], [0.7, 0.1, 0.1, 0.1]])


def test_golden_hand_cases():
    for line in open(os.path.join(GOLDEN, "verify_hand.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        v = line.split()
        toks = [int(v[0]), int(v[1])]
        n, out = ov.verify_row(P_T, P_D, toks, [float(v[2]), float(v[3])], float(v[4]))
        assert n == int(v[5])
        assert list(out) == [int(v[6]), int(v[7])]


def _first_token_distribution(p_t, p_d, M=400):
    """P(first output token = y) for gamma = 1: the draft token x drawn from
    p_d (exact weights), u_accept and u_sample integrated on midpoint grids."""
    V = len(p_t)
    us = (np.arange(M) + 0.5) / M
    dist = np.zeros(V)
    for x in range(V):
        if p_d[x] == 0:
            continue
        for u in us:
            n, out = ov.verify_row(p_t[None], p_d[None], [x], [u], 0.0)
            if n == 1:
                dist[out[0]] += p_d[x] / M
            else:
                # the resampled token depends on u_sample only: integrate it
                q = ov.quantised_weights(np.float32(p_t) - np.float32(p_d), V)
                for us_ in us:
                    dist[ov.inverse_cdf(q, us_)] += p_d[x] / M / M
    return dist


def test_output_follows_the_target_distribution():
    """The page's guarantee: whatever the draft's distribution, the token that
    comes out is distributed as p_t.  Brute force over the draft token and
    grids of both uniforms; the grid error is O(1/M)."""
    rng = np.random.default_rng(3)
    for _ in range(3):
        V = 6
        p_t = rng.dirichlet(np.ones(V))
        p_d = rng.dirichlet(np.ones(V))
        dist = _first_token_distribution(p_t, p_d, M=400)
        assert np.abs(dist - p_t).max() < 5e-3
    # a planted mistake (resampling from p_t instead of the residual) breaks it
    p_t = np.array([0.1, 0.4, 0.3, 0.2])
    p_d = np.array([0.4, 0.2, 0.2, 0.2])
    wrong = np.zeros(4)
    M = 200
    for x in range(4):
        for u in (np.arange(M) + 0.5) / M:
            if u * p_d[x] < p_t[x]:
                wrong[x] += p_d[x] / M
            else:
                wrong += p_d[x] / M * p_t
    assert np.abs(wrong - p_t).max() > 0.02


def test_identical_distributions_always_accept():
    rng = np.random.default_rng(4)
    p = rng.dirichlet(np.ones(50), size=(3, 5))
    toks = rng.integers(0, 50, size=(3, 5))
    u = rng.uniform(0, 1, size=(3, 5)) * 0.999999
    n, out = ov.verify(p, p, toks, u, rng.uniform(0, 1, size=3))
    assert np.all(n == 5) and np.array_equal(out, toks)


def test_resample_never_draws_where_draft_covers_target():
    """Tokens with p_t <= p_d have zero residual and are never resampled."""
    rng = np.random.default_rng(5)
    for _ in range(50):
        p_t = rng.dirichlet(np.ones(20))
        p_d = rng.dirichlet(np.ones(20))
        x = int(np.argmax(p_d - p_t))    # p_t < p_d here: rejection possible
        n, out = ov.verify_row(p_t[None], p_d[None], [x], [0.999999], rng.uniform())
        assert n == 0 and p_t[out[0]] > p_d[out[0]]


def test_inverse_cdf_is_bisect():
    """On the exact integer weights the draw is the standard library's
    bisect_right of the threshold in the running sums."""
    import bisect
    import itertools
    rng = np.random.default_rng(6)
    for _ in range(100):
        w = (rng.uniform(0, 1, size=30) * (rng.uniform(size=30) < 0.6)).astype(np.float32)
        q = ov.quantised_weights(w, 30)
        if sum(q) == 0:
            continue
        u = np.float32(rng.uniform())
        c = list(itertools.accumulate(q))
        t = (int(np.floor(float(u) * 2 ** 24)) * c[-1]) >> 24
        assert ov.inverse_cdf(q, u) == bisect.bisect_right(c, t)


def test_quantised_weights_keep_the_distribution():
    """The quantisation moves each weight by less than 2^-(62 - bitlen(V))."""
    rng = np.random.default_rng(7)
    V = 151936
    w = rng.dirichlet(np.ones(V)).astype(np.float32)
    q = ov.quantised_weights(w, V)
    s = 62 - V.bit_length()
    err = np.abs(np.array(q, dtype=np.float64) * 2.0 ** -s - w.astype(np.float64))
    assert err.max() < 2.0 ** -s and sum(q) < 2 ** 63
