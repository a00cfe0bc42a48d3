"""Pins of the oracle's sampling verification (T > 0) against what the
mathematics fixes: inverse-CDF buckets, the speculative-sampling theorem
(whatever the draft distribution, each emitted token follows the target's),
the acceptance rate sum_x min(p, q), and the greedy limit."""
import itertools

import numpy as np
import pytest
from scipy import stats

import oracle as O


def test_sample_from_buckets():
    w = [1.0, 2.0, 0.0, 5.0]            # running sums 1, 3, 3, 8 (exact in binary)
    cases = {0.0: 0, 0.1249: 0, 0.125: 1, 0.3749: 1, 0.375: 3, 0.5: 3, 0.9999: 3}
    for u, want in cases.items():
        assert O.sample_from(w, u) == want, u
        assert O.sample_from(np.array(w) * 37.5, u) == want, u   # unnormalised weights
    assert O.sample_from([0, 0, 5.0, 0], 0.99) == 2               # zero weights are never drawn


def test_sample_from_frequencies():
    rng = np.random.default_rng(0)
    w = rng.random(7) ** 3
    n = 60000
    draws = [O.sample_from(w, u) for u in rng.random(n)]
    counts = np.bincount(draws, minlength=7)
    assert stats.chisquare(counts, n * w / w.sum()).pvalue > 1e-4


def test_softmax_t():
    z = np.array([[1.0, 2.0, 3.0], [0.0, 0.0, 0.0]])
    np.testing.assert_allclose(O.softmax_t(z, 1.0).sum(-1), 1.0)
    np.testing.assert_allclose(O.softmax_t(z, 1.0)[0], np.exp([1, 2, 3]) / np.exp([1, 2, 3]).sum())
    np.testing.assert_allclose(O.softmax_t(z, 0.5)[0], O.softmax_t(2 * z, 1.0)[0])
    np.testing.assert_allclose(O.softmax_t(z, 3.0)[1], [1 / 3] * 3)
    with pytest.raises(ValueError):
        O.softmax_t(z, 0.0)


def _dist(rng, V, sharp=1.0):
    w = rng.random(V) ** (1 + 3 * sharp)
    return w / w.sum()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_emitted_token_follows_target(seed):
    """B = 2: one draft d ~ q, then verification.  The first emitted token
    (d if accepted, else a residual draw) must follow p exactly; when d is
    accepted the bonus must follow p[1].  A dropped clamp, a missing
    renormalisation, a residual from the wrong position or an unconditional
    accept all move these distributions."""
    rng = np.random.default_rng(seed)
    V, n = 6, 40000
    p = np.stack([_dist(rng, V), _dist(rng, V)])
    q = _dist(rng, V, sharp=0.3)[None]
    first = np.zeros(V, dtype=np.int64)
    bonus = np.zeros(V, dtype=np.int64)
    for _ in range(n):
        d = O.sample_from(q[0], rng.random())
        acc, tok, out, _ = O.verify_rejection(np.array([[0, d]]), q[None], p[None],
                                              rng.random((1, 1)), rng.random(1), np.array([0]))
        first[out[0, 0]] += 1
        if acc[0] == 1:
            bonus[out[0, 1]] += 1
    assert stats.chisquare(first, n * p[0]).pvalue > 1e-4
    m = bonus.sum()
    assert stats.chisquare(bonus, m * p[1]).pvalue > 1e-4
    # acceptance rate sum_x min(p(x), q(x)), within 4 sigma
    r = O.acceptance_probability(p[0], q[0])
    assert abs(m / n - r) < 4 * np.sqrt(r * (1 - r) / n)


def test_second_position_follows_target():
    """B = 3: the second emitted token, given the first draft accepted,
    follows p[1] whatever q[1] is."""
    rng = np.random.default_rng(7)
    V, n = 5, 40000
    p = np.stack([_dist(rng, V) for _ in range(3)])
    q = np.stack([_dist(rng, V, 0.2) for _ in range(2)])
    second = np.zeros(V, dtype=np.int64)
    for _ in range(n):
        d = [0, O.sample_from(q[0], rng.random()), O.sample_from(q[1], rng.random())]
        acc, _, out, _ = O.verify_rejection(np.array([d]), q[None], p[None], rng.random((1, 2)),
                                            rng.random(1), np.array([0]))
        if acc[0] >= 1:
            second[out[0, 1]] += 1
    assert stats.chisquare(second, second.sum() * p[1]).pvalue > 1e-4


def test_equal_distributions_accept_everything():
    rng = np.random.default_rng(3)
    V, B = 9, 6
    p = np.stack([_dist(rng, V) for _ in range(B)])
    for _ in range(200):
        d = [0] + [O.sample_from(p[j], rng.random()) for j in range(B - 1)]
        acc, _, out, new_len = O.verify_rejection(np.array([d]), p[None, :B - 1], p[None],
                                                  rng.random((1, B - 1)), rng.random(1),
                                                  np.array([10]))
        assert acc[0] == B - 1 and new_len[0] == 10 + B
        assert list(out[0, :B - 1]) == d[1:]


def test_one_hot_distributions_reduce_to_greedy():
    """T -> 0: one-hot q at the draft ids and one-hot p at the target's
    argmax give exactly verify_greedy, for every draft/posterior pair of a
    tiny B and V (exhaustive) and any uniforms."""
    rng = np.random.default_rng(5)
    V, B = 3, 4
    eye = np.eye(V)
    for draft_tail in itertools.product(range(V), repeat=B - 1):
        for post in itertools.product(range(V), repeat=B):
            draft = np.array([[1] + list(draft_tail)])
            q = eye[list(draft_tail)][None]
            p = eye[list(post)][None]
            g = O.verify_greedy(draft, np.array([post]), np.array([5]))
            r = O.verify_rejection(draft, q, p, rng.random((1, B - 1)), rng.random(1),
                                   np.array([5]))
            for a, b in zip(g, r):
                np.testing.assert_array_equal(a, b)
