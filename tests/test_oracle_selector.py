"""Pins of the oracle's DFlash 2 candidate selector (txtmix source reading,
§13-§14): top-k order against brute force, the reductions of the greedy
walk to the plain argmax, a planted bigram chain, and relabelling."""
import numpy as np
import pytest

import oracle as O


def _brute_topk(row, k):
    """Repeated argmax, lowest index first, removing each pick."""
    row = np.array(row, dtype=np.float64)
    out = []
    for _ in range(k):
        best = None
        for i, v in enumerate(row):
            if np.isnan(v):
                continue
            if best is None or v > row[best]:
                best = i
        out.append(best)
        row[best] = np.nan
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    V, k = 40, 7
    z = rng.integers(-3, 4, size=(5, V)).astype(np.float64)   # many ties
    got = O.topk_lowest(z, k)
    for r in range(5):
        assert list(got[r]) == _brute_topk(z[r], k)


def _weights(rng, V, D, r, n):
    return (rng.standard_normal((n, V)) * 2, rng.standard_normal((n, D)),
            rng.standard_normal((r, D)) * 0.2, rng.standard_normal((V, r)),
            rng.standard_normal((V, r)))


def test_k1_is_argmax():
    rng = np.random.default_rng(1)
    z, h, Wh, A, Bc = _weights(rng, 64, 16, 8, 7)
    path, cand, _ = O.select_candidates(z, h, 3, Wh, A, Bc, top_k=1)
    np.testing.assert_array_equal(path, O.argmax_lowest(z))
    np.testing.assert_array_equal(cand[:, 0], O.argmax_lowest(z))


@pytest.mark.parametrize("zero", ["pred", "succ", "gate"])
def test_vanishing_pair_term_is_argmax(zero):
    rng = np.random.default_rng(2)
    z, h, Wh, A, Bc = _weights(rng, 64, 16, 8, 9)
    if zero == "pred":
        A = np.zeros_like(A)
    elif zero == "succ":
        Bc = np.zeros_like(Bc)
    else:
        Wh = np.zeros_like(Wh)
    path, _, best = O.select_candidates(z, h, 5, Wh, A, Bc, top_k=16)
    np.testing.assert_array_equal(path, O.argmax_lowest(z))
    np.testing.assert_allclose(best, z.max(axis=1))


def _chain_case(rng, V=50, n=6, k=8, strength=40.0):
    """Codebooks encoding one bigram chain anchor -> c_1 -> ... -> c_n:
    pred rows one-hot on their own id, succ row of c_t one-hot on c_{t-1},
    a gate of ones (W_h = ones / D on rows of ones); each c_t sits at rank
    3 of its position's logits, inside the top k but not on top."""
    D = r = V
    anchor = 7
    chain = rng.choice([i for i in range(V) if i != anchor], size=n, replace=False)
    z = rng.standard_normal((n, V))
    for t in range(n):
        order = np.argsort(-z[t])
        c = chain[t]
        z[t, c] = (z[t, order[2]] + z[t, order[3]]) / 2 if order[2] != c else z[t, c]
    A = np.eye(V)
    Bc = np.zeros((V, r))
    prev = anchor
    for c in chain:
        Bc[c, prev] = strength
        prev = c
    h = np.ones((n, D))
    Wh = np.ones((r, D)) / D
    return z, h, Wh, A, Bc, anchor, chain, k


def test_planted_bigram_chain_is_followed():
    rng = np.random.default_rng(3)
    z, h, Wh, A, Bc, anchor, chain, k = _chain_case(rng)
    assert all(c not in O.argmax_lowest(z)[t:t + 1] for t, c in enumerate(chain))
    path, cand, _ = O.select_candidates(z, h, anchor, Wh, A, Bc, top_k=k)
    assert all(chain[t] in cand[t] for t in range(len(chain)))
    np.testing.assert_array_equal(path, chain)
    # the two codebooks swapped: the pair term looks backwards and the chain is lost
    swapped, _, _ = O.select_candidates(z, h, anchor, Wh, Bc, A, top_k=k)
    assert not np.array_equal(swapped, chain)
    # another anchor: the chain's first link never fires, so neither do the rest
    other, _, _ = O.select_candidates(z, h, anchor + 1, Wh, A, Bc, top_k=k)
    np.testing.assert_array_equal(other, O.argmax_lowest(z))


def test_relabelling_the_vocabulary_relabels_the_path():
    rng = np.random.default_rng(4)
    V = 64
    z, h, Wh, A, Bc = _weights(rng, V, 16, 8, 10)
    perm = rng.permutation(V)            # new id of token i is perm[i]
    inv = np.argsort(perm)
    path, _, best = O.select_candidates(z, h, 11, Wh, A, Bc, top_k=6)
    path2, _, best2 = O.select_candidates(z[:, inv], h, int(perm[11]), Wh, A[inv], Bc[inv], 6)
    np.testing.assert_array_equal(path2, perm[path])
    np.testing.assert_allclose(best2, best)
