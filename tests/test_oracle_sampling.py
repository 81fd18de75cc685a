"""Pins for the sampling oracle.

The oracle's decisions are checked against what the pages prove:
  * exact enumeration: with dyadic p, q on a tiny vocabulary every (u, v) cell
    of the oracle's piecewise-constant decision is enumerated with exact
    rational measure; P(first emitted = y) must equal p(y) exactly (quant67
    section 3.2), the residual normaliser must equal 1 - sum min(p, q), and the
    number of accepted drafts must follow the truncated geometric law with the
    per-position alpha ("KV Cache + Speculative Decoding" section 7.4);
  * the two-token worked example (CS336 lecture 10 section 8, in its swapped
    naming: there the draft is p and the target q);
  * Monte-Carlo laws: E[tau] = (1 - alpha^(K+1)) / (1 - alpha) for identical
    rows, the page's sanity checks (alpha within 1 % over 100k samples; total
    variation of the output vs direct target sampling below 0.01;
    "KV Cache + Speculative Decoding" appendix A.2);
  * special cases: q = p accepts everything, one-hot p is deterministic, K = 0
    is a plain inverse-CDF draw (numpy searchsorted), softmax matches scipy.
"""
from fractions import Fraction as F

import numpy as np
import pytest
import scipy.special

from oracle import sampling, theory


# ---------------------------------------------------------------- helpers ---

def dyadic_dist(rng, V, denom=64, zeros=True):
    """Random distribution with entries k/denom (exact in binary floating point)."""
    while True:
        cuts = np.sort(rng.integers(0, denom + 1, size=V - 1))
        k = np.diff(np.concatenate([[0], cuts, [denom]]))
        if not zeros and (k == 0).any():
            continue
        if k.sum() == denom:
            return [F(int(v), denom) for v in k]


def cells(breaks):
    """Sorted distinct breakpoints in [0, 1] -> list of (lo, hi) cells."""
    pts = sorted(set([F(0), F(1)] + [b for b in breaks if 0 < b < 1]))
    return [(pts[i], pts[i + 1]) for i in range(len(pts) - 1)]


def cdf_breaks(w):
    Z = sum(w)
    c, out = F(0), []
    for wi in w:
        c += wi
        out.append(c / Z)
    return out


def enumerate_round(P, Q):
    """Exact law of the oracle's output for fixed rows P[0..K], Q[0..K-1].

    Returns {(num_accepted, tuple(out_tokens)): Fraction}.
    """
    K, V = len(Q), len(P[0])
    # phase 1: draft tokens x and the u cells decide the sampled row n
    cases = []
    for flat in range(V ** K):
        x = [(flat // V ** i) % V for i in range(K)]
        wx = F(1)
        for i in range(K):
            wx *= Q[i][x[i]]
        if wx == 0:
            continue
        u_cells_per_pos = []
        for i in range(K):
            r = min(F(1), P[i][x[i]] / Q[i][x[i]])
            u_cells_per_pos.append(cells([r]))
        # product of u cells
        idx = [0] * K
        while True:
            cell = [u_cells_per_pos[i][idx[i]] for i in range(K)]
            wu = F(1)
            for lo, hi in cell:
                wu *= hi - lo
            umid = [(lo + hi) / 2 for lo, hi in cell]
            cases.append((x, umid, wx * wu))
            j = 0
            while j < K:
                idx[j] += 1
                if idx[j] < len(u_cells_per_pos[j]):
                    break
                idx[j] = 0
                j += 1
            if j == K:
                break
    p_arr = np.array([[float(v) for v in row] for row in P])[None]
    q_arr = np.array([[float(v) for v in row] for row in Q]).reshape(1, K, V)
    law = {}
    for x, umid, w in cases:
        uni = np.full((1, K + 1, 2), 0.5)
        for i in range(K):
            uni[0, i, 0] = float(umid[i])
        r1 = sampling.verify_from_probs(p_arr, q_arr, np.array([x]), uni)
        n = int(r1["num_accepted"][0])
        if n < K:
            wts = [max(F(0), P[n][y] - Q[n][y]) for y in range(V)]
        else:
            wts = list(P[K])
        for lo, hi in cells(cdf_breaks(wts)):
            uni2 = uni.copy()
            uni2[0, n, 1] = float((lo + hi) / 2)
            r = sampling.verify_from_probs(p_arr, q_arr, np.array([x]), uni2)
            assert int(r["num_accepted"][0]) == n
            key = (n, tuple(int(t) for t in r["out_tokens"][0]))
            law[key] = law.get(key, F(0)) + w * (hi - lo)
    return law


def alpha_exact(p, q):
    return sum(min(a, b) for a, b in zip(p, q))


# ------------------------------------------------------- exact enumeration ---

@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("V", [2, 3, 4, 5])
def test_single_position_output_law_is_exactly_p(seed, V):
    rng = np.random.default_rng(1000 * V + seed)
    p1, q1, p2 = dyadic_dist(rng, V), dyadic_dist(rng, V), dyadic_dist(rng, V)
    law = enumerate_round([p1, p2], [q1])
    assert sum(law.values()) == 1
    first = [F(0)] * V
    second = [F(0)] * V
    n_law = [F(0), F(0)]
    for (n, toks), w in law.items():
        first[toks[0]] += w
        n_law[n] += w
        if n == 1:
            second[toks[1]] += w
            assert toks[0] == toks[0]
        else:
            assert toks[1] == -1
    assert first == p1                                   # P(output = y) = p(y)
    a = alpha_exact(p1, q1)
    assert n_law == [1 - a, a]
    assert second == [a * v for v in p2]                 # bonus ~ p_{K+1}


@pytest.mark.parametrize("seed", range(6))
def test_two_positions_truncated_geometric_and_marginals(seed):
    rng = np.random.default_rng(77 + seed)
    V = 3
    P = [dyadic_dist(rng, V) for _ in range(3)]
    Q = [dyadic_dist(rng, V) for _ in range(2)]
    law = enumerate_round(P, Q)
    assert sum(law.values()) == 1
    a1, a2 = alpha_exact(P[0], Q[0]), alpha_exact(P[1], Q[1])
    n_law = [F(0)] * 3
    first = [F(0)] * V
    second = [F(0)] * V
    third = [F(0)] * V
    for (n, toks), w in law.items():
        n_law[n] += w
        first[toks[0]] += w
        if n >= 1:
            second[toks[1]] += w
        if n >= 2:
            third[toks[2]] += w
        assert all(t == -1 for t in toks[n + 1:])
    assert n_law == [1 - a1, a1 * (1 - a2), a1 * a2]
    assert first == P[0]
    assert second == [a1 * v for v in P[1]]
    assert third == [a1 * a2 * v for v in P[2]]


def test_disjoint_supports_and_zero_draft_mass():
    # the draft never proposes what the target wants: every draft is rejected
    # and the residual is p itself
    P = [[F(1, 2), F(1, 2), F(0), F(0)], [F(1, 4)] * 4]
    Q = [[F(0), F(0), F(1, 2), F(1, 2)]]
    law = enumerate_round(P, Q)
    assert {k: v for k, v in law.items()} == {(0, (0, -1)): F(1, 2), (0, (1, -1)): F(1, 2)}


def test_residual_mass_equals_one_minus_alpha_exactly():
    rng = np.random.default_rng(5)
    for _ in range(200):
        V = int(rng.integers(2, 9))
        p, q = dyadic_dist(rng, V, 256), dyadic_dist(rng, V, 256)
        Z = sum(max(F(0), a - b) for a, b in zip(p, q))
        assert Z == 1 - alpha_exact(p, q)
        # the oracle's own float computation of the residual mass is exact here
        pa = np.array([[[float(v) for v in p], [1.0] + [0.0] * (V - 1)]])
        qa = np.array([[[float(v) for v in q]]])
        x = np.array([[int(np.argmax(qa[0, 0]))]])
        uni = np.array([[[0.999999, 0.5], [0.5, 0.5]]])
        r = sampling.verify_from_probs(pa, qa, x, uni)
        if r["num_accepted"][0] == 0 and Z > 0:
            assert r["sampled_mass"][0] == float(Z)
        assert theory.alpha(pa[0, 0], qa[0, 0]) == float(alpha_exact(p, q))
        assert theory.alpha_from_l1(pa[0, 0], qa[0, 0]) == pytest.approx(float(alpha_exact(p, q)), abs=1e-15)


def test_two_token_worked_example_renamed():
    # CS336 lecture 10, section 8: two-token vocabulary {A, B}, the draft
    # over-weights A. Renamed to p = target, q = draft: q(A) > p(A).
    p = [F(1, 4), F(3, 4)]
    q = [F(3, 4), F(1, 4)]
    law = enumerate_round([p, [F(1, 2), F(1, 2)]], [q])
    first = [F(0), F(0)]
    for (n, toks), w in law.items():
        first[toks[0]] += w
    # P(A) = q(A) * p(A)/q(A) = p(A); P(B) = q(B)*1 + q(A)*(1 - p(A)/q(A)) = p(B)
    assert first == p
    assert first[0] == q[0] * (p[0] / q[0])
    assert first[1] == q[1] + q[0] * (1 - p[0] / q[0])


# ------------------------------------------------ strictness at boundaries ---

def test_accept_boundary_is_strict():
    p = np.array([[[0.25, 0.75], [0.5, 0.5]]])
    q = np.array([[[0.5, 0.5]]])
    x = np.array([[0]])
    # ratio p/q = 0.5: u = 0.5 rejects, u just below accepts
    r = sampling.verify_from_probs(p, q, x, np.array([[[0.5, 0.3], [0.0, 0.3]]]))
    assert r["num_accepted"][0] == 0
    r = sampling.verify_from_probs(p, q, x, np.array([[[np.nextafter(0.5, 0), 0.3], [0.0, 0.3]]]))
    assert r["num_accepted"][0] == 1


def test_inverse_cdf_strict_and_skips_zero_weight():
    w = np.array([[0.25, 0.0, 0.25, 0.5]])
    # v*Z exactly at C(0) = 0.25: strict '>' moves past token 0 and skips the
    # zero-weight token 1
    y, _, _ = sampling.inverse_cdf(w, np.array([0.25]))
    assert y[0] == 2
    y, _, _ = sampling.inverse_cdf(w, np.array([0.0]))
    assert y[0] == 0
    y, _, _ = sampling.inverse_cdf(np.array([[0.5, 0.5, 0.0, 0.0]]), np.array([0.9999999999]))
    assert y[0] == 1


def test_inverse_cdf_matches_searchsorted():
    rng = np.random.default_rng(3)
    for _ in range(50):
        V = int(rng.integers(1, 300))
        w = rng.random(V) * (rng.random(V) < 0.7)
        if w.sum() == 0:
            w[0] = 1.0
        v = rng.random()
        C = np.cumsum(w)
        ref = int(np.searchsorted(C, v * C[-1], side="right"))
        y, margin, Z = sampling.inverse_cdf(w[None], np.array([v]))
        assert y[0] == ref
        assert Z[0] == C[-1]
        assert 0 <= margin[0] <= 1


# ---------------------------------------------------------- special cases ---

def test_q_equal_p_accepts_all_and_bonus_from_last_row():
    rng = np.random.default_rng(11)
    B, K, V = 64, 5, 50
    logits = rng.normal(0, 3, size=(B, K + 1, V))
    x = rng.integers(0, V, size=(B, K))
    uni = rng.random((B, K + 1, 2))
    r = sampling.rejection_sample(logits, logits[:, :K], x, uni)
    assert (r["num_accepted"] == K).all()
    p_last = scipy.special.softmax(logits[:, K], axis=1)
    for b in range(B):
        C = np.cumsum(p_last[b])
        assert r["out_tokens"][b, K] == np.searchsorted(C, uni[b, K, 1] * C[-1], side="right")
        assert (r["out_tokens"][b, :K] == x[b]).all()


def test_one_hot_target_is_deterministic():
    V, K = 10, 3
    logits = np.full((1, K + 1, V), -1e4)
    logits[0, :, 7] = 0.0
    draft = np.zeros((1, K, V))
    for x0 in range(V):
        x = np.array([[x0, 7, 7]])
        for u in [0.0, 0.3, 0.99]:
            uni = np.full((1, K + 1, 2), u)
            r = sampling.rejection_sample(logits, draft, x, uni)
            if x0 == 7:
                assert r["num_accepted"][0] == K and list(r["out_tokens"][0]) == [7, 7, 7, 7]
            else:
                assert r["num_accepted"][0] == 0 and list(r["out_tokens"][0]) == [7, -1, -1, -1]


def test_k_zero_is_plain_inverse_cdf():
    rng = np.random.default_rng(2)
    B, V = 32, 100
    logits = rng.normal(0, 3, size=(B, 1, V))
    uni = rng.random((B, 1, 2))
    r = sampling.rejection_sample(logits, np.zeros((B, 0, V)), np.zeros((B, 0), dtype=np.int64), uni)
    p = scipy.special.softmax(logits[:, 0], axis=1)
    for b in range(B):
        C = np.cumsum(p[b])
        assert r["out_tokens"][b, 0] == np.searchsorted(C, uni[b, 0, 1] * C[-1], side="right")
    assert (r["num_accepted"] == 0).all()


@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_softmax_matches_scipy(T):
    rng = np.random.default_rng(4)
    x = rng.normal(0, 3, size=(5, 3, 1000))
    assert np.allclose(sampling.softmax(x, T), scipy.special.softmax(x / T, axis=-1), rtol=1e-13, atol=0)


# ------------------------------------------------------------ Monte-Carlo ---

def _mc_round(rng, p_row, q_row, K, N):
    V = len(p_row)
    P = np.broadcast_to(p_row, (N, K + 1, V))
    Q = np.broadcast_to(q_row, (N, K, V))
    x = rng.choice(V, size=(N, K), p=q_row)
    uni = rng.random((N, K + 1, 2))
    return sampling.verify_from_probs(P, Q, x, uni)


@pytest.mark.parametrize("K", [1, 4, 7])
def test_monte_carlo_expected_tokens(K):
    rng = np.random.default_rng(100 + K)
    V, N = 8, 200_000
    p_row = rng.dirichlet(np.ones(V))
    q_row = 0.6 * p_row + 0.4 * rng.dirichlet(np.ones(V))
    a = theory.alpha(p_row, q_row)
    r = _mc_round(rng, p_row, q_row, K, N)
    emitted = r["num_accepted"] + 1
    se = emitted.std() / np.sqrt(N)
    assert abs(emitted.mean() - theory.expected_tokens(a, K)) < 4 * se
    # and the whole length law is the truncated geometric one
    pmf = theory.accepted_length_pmf([a] * K)
    counts = np.bincount(r["num_accepted"], minlength=K + 1) / N
    assert np.all(np.abs(counts - pmf) < 4 * np.sqrt(np.array(pmf) * (1 - np.array(pmf)) / N) + 1e-12)


def test_page_sanity_checks_alpha_and_tv():
    # "KV Cache + Speculative Decoding" appendix A.2: alpha estimated over 100k
    # samples within 1 % of theory; spec output vs direct target sampling TV < 0.01
    rng = np.random.default_rng(9)
    V, N, K = 8, 100_000, 4
    p_row = rng.dirichlet(np.ones(V) * 2)
    q_row = 0.5 * p_row + 0.5 * rng.dirichlet(np.ones(V) * 2)
    a = theory.alpha(p_row, q_row)
    r = _mc_round(rng, p_row, q_row, K, N)
    a_hat = (r["num_accepted"] >= 1).mean()
    assert abs(a_hat - a) / a < 0.01
    first = np.bincount(r["out_tokens"][:, 0], minlength=V) / N
    assert 0.5 * np.abs(first - p_row).sum() < 0.01
