"""Pins of the tree rejection-sampling oracle.

- A chain given as a tree (node j + 1 is draft j, drafted from row j) gives
  the chain oracle's tokens and accepted lengths exactly (uniform indices
  mapped: node j + 1 takes draft j's accept uniform, node j the draw of row
  j).
- The reading's exactness, by exact enumeration with Fractions: siblings
  drawn i.i.d. from q_u and tried in turn against the running residual give
  a first emitted token distributed exactly as p_u, for any p and q (the
  property that makes recursive rejection exact; it fails for a plain
  "retry with p" rule, which the same enumeration shows).
- The oracle's code against that law: Monte Carlo over random uniforms and
  i.i.d. sibling tokens, within 4.5 sigma per token.
"""
from fractions import Fraction as F

import numpy as np
import pytest

from oracle import sampling


def chain_case(rng, B, K, V):
    tl = rng.normal(0, 2, (B, K + 1, V))
    dl = tl[:, :K] + rng.normal(0, 1, (B, K, V))
    q = sampling.softmax(dl)
    tok = np.array([[rng.choice(V, p=q[b, i]) for i in range(K)] for b in range(B)])
    uv = rng.uniform(0, 1, (B, K + 1, 2))
    return tl, dl, tok, uv


@pytest.mark.parametrize("seed", range(6))
def test_chain_tree_is_the_chain(seed):
    rng = np.random.default_rng(seed)
    B, K, V = 16, int(rng.integers(1, 6)), int(rng.integers(3, 40))
    tl, dl, tok, uv = chain_case(rng, B, K, V)
    ref = sampling.rejection_sample(tl, dl, tok, uv)
    n = K + 1
    parent = np.tile(np.arange(-1, n - 1), (B, 1))
    ttok = np.concatenate([np.zeros((B, 1), dtype=np.int64), tok], axis=1)
    tdraft = np.concatenate([dl, np.zeros((B, 1, V))], axis=1)       # the leaf's row is unused
    tuv = np.empty((B, n, 2))
    tuv[:, 1:, 0] = uv[:, :K, 0]
    tuv[:, 0, 0] = 0.5
    tuv[:, :, 1] = uv[:, :, 1]
    got = sampling.tree_rejection_sample(tl, tdraft, parent, ttok, tuv)
    assert np.array_equal(got["num_accepted"], ref["num_accepted"])
    assert np.array_equal(got["out_tokens"], ref["out_tokens"])
    for b in range(B):
        assert list(got["path_nodes"][b, :ref["num_accepted"][b]]) == list(range(1, ref["num_accepted"][b] + 1))


@pytest.mark.parametrize("seed", range(4))
def test_decision_record_of_a_chain_matches_the_chain_oracle(seed):
    # the walk's decision list against the chain oracle's own record: one
    # accept test per visited draft (its margin |u - p/q| and outcome), then
    # the draw at the last node with its CDF margin and the emitted token
    rng = np.random.default_rng(100 + seed)
    B, K, V = 12, int(rng.integers(1, 5)), int(rng.integers(3, 30))
    tl, dl, tok, uv = chain_case(rng, B, K, V)
    ref = sampling.rejection_sample(tl, dl, tok, uv)
    n = K + 1
    parent = np.tile(np.arange(-1, n - 1), (B, 1))
    ttok = np.concatenate([np.zeros((B, 1), dtype=np.int64), tok], axis=1)
    tdraft = np.concatenate([dl, np.zeros((B, 1, V))], axis=1)
    tuv = np.empty((B, n, 2))
    tuv[:, 1:, 0] = uv[:, :K, 0]
    tuv[:, 0, 0] = 0.5
    tuv[:, :, 1] = uv[:, :, 1]
    got = sampling.tree_rejection_sample(tl, tdraft, parent, ttok, tuv)
    for b in range(B):
        dec = got["decisions"][b]
        na = int(ref["num_accepted"][b])
        tests = dec[:-1]
        assert len(tests) == min(na + 1, K)
        for i, (u, c, m, outcome) in enumerate(tests):
            assert (u, c) == (i, i + 1)
            assert outcome == (i < na)
            assert m == pytest.approx(ref["accept_margin"][b, i], rel=1e-12, abs=1e-15)
        u, c, m, y = dec[-1]
        assert (u, c) == (na, -1)
        assert y == ref["out_tokens"][b, na]
        assert m == pytest.approx(ref["cdf_margin"][b], rel=1e-9, abs=1e-15)
        assert got["margin"][b] == min(d[2] for d in dec)


def first_token_law(p, q, k, residual=True):
    """Exact law of the first emitted token when k siblings are drawn i.i.d.
    from q and tried in turn (each sibling a leaf: an accepted one is the
    emitted token). residual=False retries every sibling against p itself."""
    V = len(p)
    law = [F(0)] * V

    def walk(r, left, weight):
        if left == 0:
            for y in range(V):
                law[y] += weight * r[y]
            return
        for x in range(V):
            if q[x] == 0:
                continue
            acc = min(F(1), r[x] / q[x])
            law[x] += weight * q[x] * acc
            if acc < 1:
                if residual:
                    res = [max(F(0), r[i] - q[i]) for i in range(V)]
                    z = sum(res)
                    nr = [v / z for v in res] if z > 0 else list(p)
                else:
                    nr = list(p)
                walk(nr, left - 1, weight * q[x] * (1 - acc))

    walk(list(p), k, F(1))
    return law


@pytest.mark.parametrize("k", [1, 2, 3])
@pytest.mark.parametrize("case", range(4))
def test_sibling_rule_is_exact(k, case):
    rng = np.random.default_rng(100 + case)
    V = 3 + case % 2
    p = [F(int(a), 64) for a in rng.multinomial(64, np.ones(V) / V)]
    q = [F(int(a), 64) for a in rng.multinomial(64, np.ones(V) / V)]
    assert first_token_law(p, q, k) == p


def test_retrying_against_p_is_not_exact():
    p = [F(1, 2), F(1, 4), F(1, 4)]
    q = [F(1, 8), F(3, 4), F(1, 8)]
    assert first_token_law(p, q, 2, residual=True) == p
    assert first_token_law(p, q, 2, residual=False) != p


def test_oracle_sibling_law_monte_carlo():
    rng = np.random.default_rng(7)
    V, N = 4, 40000
    p = np.array([0.45, 0.3, 0.15, 0.1])
    q = np.array([0.1, 0.2, 0.3, 0.4])
    # root with three leaf children; logits are log-probabilities
    tl = np.tile(np.log(p), (N, 4, 1))
    dl = np.tile(np.log(q), (N, 4, 1))
    parent = np.tile(np.array([-1, 0, 0, 0]), (N, 1))
    tok = np.zeros((N, 4), dtype=np.int64)
    tok[:, 1:] = rng.choice(V, size=(N, 3), p=q)
    uv = rng.uniform(0, 1, (N, 4, 2))
    got = sampling.tree_rejection_sample(tl, dl, parent, tok, uv)
    first = got["out_tokens"][:, 0]
    freq = np.bincount(first, minlength=V) / N
    sigma = np.sqrt(p * (1 - p) / N)
    assert np.all(np.abs(freq - p) < 4.5 * sigma), (freq, p)


def test_siblings_are_tried_in_bfs_order_by_hand():
    # q = p, so every child is accepted: the first child in BFS order wins
    # (token 2 of node 1), then node 1 is a leaf and its row (one-hot on
    # token 0) gives the bonus
    V = 3
    tl = np.log(np.array([[[1 / 3, 1 / 3, 1 / 3], [1.0, 1e-30, 1e-30], [1e-30, 1.0, 1e-30]]]))
    dl = tl.copy()
    got = sampling.tree_rejection_sample(tl, dl, np.array([[-1, 0, 0]]), np.array([[0, 2, 1]]),
                                         np.full((1, 3, 2), 0.5))
    assert got["num_accepted"][0] == 1
    assert list(got["path_nodes"][0]) == [1, -1, -1]
    assert list(got["out_tokens"][0]) == [2, 0, -1]


# ---- typical acceptance (the Medusa rule, opt-in and not exact) ----

def test_entropy_matches_scipy():
    import scipy.stats
    rng = np.random.default_rng(4)
    p = rng.dirichlet(np.ones(50), size=6)
    p[0, :10] = 0
    p[0] /= p[0].sum()
    assert np.allclose(sampling.entropy(p), scipy.stats.entropy(p, axis=-1), rtol=1e-12, atol=0)


def test_typical_threshold_by_hand():
    # uniform p over V: H = ln V, tau = min(eps, delta / V); a draft is accepted
    # iff 1/V > tau
    V = 8
    tl = np.zeros((2, 2, V))
    dl = np.zeros((2, 2, V))
    par = np.array([[-1, 0], [-1, 0]])
    tok = np.array([[0, 3], [0, 3]])
    uv = np.full((2, 2, 2), 0.5)
    acc = sampling.tree_rejection_sample(tl, dl, par, tok, uv, typical=(0.3, 0.9))   # tau = 0.1125 < 0.125
    rej = sampling.tree_rejection_sample(tl, dl, par, tok, uv, typical=(0.3, 1.1))   # tau = 0.1375 > 0.125
    assert list(acc["num_accepted"]) == [1, 1] and list(acc["out_tokens"][0]) == [3, 4]
    assert list(rej["num_accepted"]) == [0, 0] and list(rej["out_tokens"][0]) == [4, -1]


def test_typical_never_accepting_draws_from_p():
    # tau = min(1, huge) = 1 is never exceeded: the first token is drawn from
    # p_root itself (no residual), so its law is p_root (Monte Carlo)
    rng = np.random.default_rng(5)
    V, N = 5, 30000
    p = np.array([0.4, 0.25, 0.2, 0.1, 0.05])
    tl = np.tile(np.log(p), (N, 3, 1))
    par = np.tile(np.array([-1, 0, 0]), (N, 1))
    tok = np.zeros((N, 3), dtype=np.int64)
    tok[:, 1:] = rng.integers(0, V, (N, 2))
    uv = rng.uniform(0, 1, (N, 3, 2))
    got = sampling.tree_rejection_sample(tl, tl.copy(), par, tok, uv, typical=(1.0, 1e9))
    assert (got["num_accepted"] == 0).all()
    freq = np.bincount(got["out_tokens"][:, 0], minlength=V) / N
    assert np.all(np.abs(freq - p) < 4.5 * np.sqrt(p * (1 - p) / N))
